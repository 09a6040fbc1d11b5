// Decode over the paged cache on the tensor core: one query token per
// sequence (paged_attn_decode), or a uniform batch of q tokens per sequence
// (paged_attn_decode_multi, speculative decoding).
//
// What is computed (xformers.py XFormersImpl.forward -> forward_decode;
// cpu_attn TorchSDPABackendImpl.forward -> forward_decode; for q > 1
// backends.utils AttentionCGSupport.UNIFORM_BATCH: every decode of the batch
// has the same query length q = 1 + num_speculative_tokens, and
// AttentionMetadataBuilder._init_reorder_batch_threshold pulls such decodes
// to the front for spec-as-decode kernels): token t of sequence b sits at
// position i = L_b - q + t (L_b counts the q new tokens, as a single-token
// decode's seq_len counts its one) and attends to keys lo(i) <= j <= i read
// through the block table:
//     s_j = scale * q.k_j + slope_h * (j - i),   out = softmax(s) . V.
//
// Design.  Rows are (token t, query head h of the KV group) pairs,
// r = t * QPK + h, in groups of 16: one m16 tile of mma.sync m16n8k16, so the
// group's rows share every K/V byte.  (tcgen05's smallest tile, 64 rows,
// would leave most of it empty at these row counts; the step is bound by
// HBM, and the tensor core serves to keep the per-key instruction count low
// enough for the 8-bit cache's doubled key rate.)  CTA = (split of the key
// range, KV head x row group, sequence), 4 warps.  Each warp walks its own
// 16-token units of the split (unit k of the warp = split unit warp + 4k)
// through a two-stage ring of TMA boxes (16 tokens x 64 dims, 128-byte
// swizzle; K and V).  Per unit:
//   S[16 rows x 16 keys] = Q K^T   Q fragments held in registers for the
//                                  whole CTA, K fragments by ldmatrix;
//   scores scaled into the log2 domain (+ ALiBi), masked per row (its own
//   causal position and window start), online softmax per row with a lazy
//   reference max (moved, and O rescaled, only when a score passes it by 2^8);
//   O += P V                       P packed to bf16/fp16 pairs in registers as
//                                  the A operand, V fragments by
//                                  ldmatrix.trans.
// The four warps merge their (m, l, O) through shared memory; a sequence cut
// into several splits writes (o, m, l) partials that decode_combine_kernel
// merges (flash-decoding).  Every wait is bounded (a timeout records
// PKV_ERR_TIMEOUT, drains the warp's copies in flight and leaves the output
// unwritten for that CTA).
//
// Over an fp8 (E4M3) cache (KV8) the boxes carry the 8-bit codes (16 tokens x
// D bytes, 128-byte swizzle; 64-byte for D = 64).  q.k runs on the codes as
// they are: mma.sync m16n8k32 on E4M3 operands, each query row scaled by a
// power of two 2^-e (e from the row group's largest magnitude, largest
// |q| in [2^7, 2^8)) and split into two E4M3 terms hi + lo, which hold every
// component within 2^10 of the largest exactly (a bf16 value has 8
// significant bits; hi takes 4, the remainder fits lo's 4); the head
// dimension is taken in a fixed permuted order (lane tq of k-step s covers
// dims tq * D/4 + 8s .. + 7, its own 16-byte chunk of each key row) that the
// query fragments follow too (a dot product does not depend on the order of
// its terms).  p.V runs transposed, O^T += V^T P^T on fp16 operands: the
// P fragments of the score tile are already the B operand, and a lane builds
// its V^T fragments from the codes of keys 2tq, 2tq+1, 2tq+8, 2tq+9 (its
// dims 16g .. 16g+15, one 16-byte chunk per key row) with byte permutes and
// cvt.rn.f16x2.e4m3x2, so the codes never go back to shared memory.  2^e
// and k_scale join the softmax scale, v_scale multiplies the output.
//
// Decode context parallelism (backends.utils CommonAttentionMetadata
// dcp_local_seq_lens): a rank of a group of R holds token j of each sequence
// when j % R is its rank, at local position j / R.  The same kernel runs over
// the rank's own cache and tables with local key k at position k * R + rank
// (masks, ALiBi, the mask-free test), and writes the rank's share, its fp32
// (o, m, l) per row and head, instead of the output; dcp_combine_kernel
// merges the all-gathered shares.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace dec {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kUnit = 16;   // keys per unit (one TMA box height)
constexpr int kRows = 16;   // rows per CTA: one m16 tile
// TMA ring depth per warp.  (A 3-deep ring for the fp8 cache, which moves
// half the bytes per unit, measured the same as 2: the fp8 decode is bound by
// the per-unit instruction latency of its warps, not by bytes in flight.)
template <bool KV8>
struct Ring {
  static constexpr int stages = 2;
};
constexpr float kLazy = 8.f;

struct Args {
  void *out;
  const uint16_t *query;
  const int32_t *block_tables;
  const int32_t *seq_lens;
  const float *alibi;
  float *part_o;   // [B * q * H][max_splits][D]
  float *part_ml;  // [B * q * H][max_splits][2]
  int64_t num_blocks;
  int num_seqs, max_blocks_per_seq;
  int H, QPK, q, rows, row_groups;
  int BS, window, split_units, max_splits;
  float scale_log2;  // scale * log2(e) (* k_scale over an fp8 cache)
  float v_scale;     // 1, or the fp8 cache's value scale
  // decode context parallelism: this rank holds token j of a sequence when
  // j % dcp_world == dcp_rank, at local position j / dcp_world (1, 0: off)
  int dcp_world, dcp_rank;
  // partial output (a rank's share): normalised o [rows * H][D] and (m, l)
  // [rows * H][2] in fp32 instead of `out` (null: write `out`)
  float *res_o, *res_ml;
};

struct Span {
  int L;           // length (0: padding, or a bad length that was reported)
  int first_unit;  // unit (of this rank's local tokens) of the first visible key
  int nunits;      // units up to the rank's last token (0: it holds no visible key)
  int nsplit;
};

__device__ __forceinline__ Span span_of(const Args &a, int b, bool report) {
  Span s{};
  int L = __ldg(a.seq_lens + b);
  const int R = a.dcp_world, r = a.dcp_rank;
  const int cap = a.max_blocks_per_seq * a.BS;  // local tokens the table can hold
  const int Lr = L > r ? (L - r + R - 1) / R : 0;  // this rank's tokens
  if (L < 0 || Lr > cap || (L > 0 && L < a.q)) {  // the decode must fit its sequence
    if (report) record_error(PKV_ERR_BOUNDS, b);
    L = 0;
  }
  s.L = L;
  if (L == 0) return s;
  const int i0 = L - a.q;  // token 0: its window starts first
  const int lo = a.window > 0 ? max(0, i0 - a.window + 1) : 0;
  const int first = lo > r ? (lo - r + R - 1) / R : 0;  // first local token at or past lo
  if (first >= Lr) return s;  // nothing visible on this rank: nunits = 0
  s.first_unit = first / kUnit;
  s.nunits = (Lr - 1) / kUnit - s.first_unit + 1;
  s.nsplit = (s.nunits + a.split_units - 1) / a.split_units;
  if (s.nsplit > a.max_splits) {  // seq_len above the host's max_seq_len
    if (report) record_error(PKV_ERR_BOUNDS, b);
    s.nsplit = a.max_splits;
  }
  return s;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// D[16x8] += A[16x16] B[16x8], fp32 accumulate; A row-major, B column-major.
template <class T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<BF16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<FP16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same product when only rows 0..7 of A are used (rows 8..15 zero): the
// lane's A registers of rows g + 8 are zero and the D elements of those rows
// are discarded, so a caller keeps half the fragments.
template <class T>
__device__ __forceinline__ void mma16816_top(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0,
                                             uint32_t b1);
template <>
__device__ __forceinline__ void mma16816_top<BF16>(float (&d)[2], uint32_t a0, uint32_t a2,
                                                   uint32_t b0, uint32_t b1) {
  asm volatile(
      "{\n\t.reg .f32 z0, z1;\n\t"
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, z0, z1}, "
      "{%2, %4, %3, %4}, {%5, %6}, {%0, %1, %7, %7};\n\t}"
      : "+f"(d[0]), "+f"(d[1])
      : "r"(a0), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
}
template <>
__device__ __forceinline__ void mma16816_top<FP16>(float (&d)[2], uint32_t a0, uint32_t a2,
                                                   uint32_t b0, uint32_t b1) {
  asm volatile(
      "{\n\t.reg .f32 z0, z1;\n\t"
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, z0, z1}, "
      "{%2, %4, %3, %4}, {%5, %6}, {%0, %1, %7, %7};\n\t}"
      : "+f"(d[0]), "+f"(d[1])
      : "r"(a0), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
}

template <int D, bool KV8 = false>
struct Lay {
  static constexpr int BOX = kUnit * 128;  // 16 rows x 64 dims x 2 B
  static constexpr int V16 = (D / 64) * BOX;  // one unit of K or V as 16-bit values
  static constexpr int TILE = KV8 ? kUnit * D : V16;  // one unit as stored in the cache
  static constexpr int STAGE = 2 * TILE;
  // per-warp rings, then (16-bit cache) a zero V tile; the merge buffers
  // reuse the area once the rings are drained
  static constexpr int NST = Ring<KV8>::stages;
  static constexpr int ZERO = kWarps * NST * STAGE;
  static constexpr int MERGE = kWarps * kRows * (D + 2) * 4;
  static constexpr int TILES = (ZERO + (KV8 ? 0 : V16)) > MERGE ? ZERO + (KV8 ? 0 : V16) : MERGE;
};

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Byte offset, inside a unit's tile of E4M3 codes (16 key rows of D bytes,
// loaded with the 128-byte swizzle for D = 128 and the 64-byte one for
// D = 64), of 16-byte chunk `chunk` of key row `row`.
template <int D>
__device__ __forceinline__ uint32_t swz8(int row, int chunk) {
  if constexpr (D == 128)
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
  else
    return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// D[16x8] += A[16x32] B[32x8] on E4M3 operands, fp32 accumulate.
__device__ __forceinline__ void mma16832_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The same with rows 8..15 of A zero (their results discarded).
__device__ __forceinline__ void mma16832_e4m3_top(float (&d)[2], uint32_t a0, uint32_t a2,
                                                  uint32_t b0, uint32_t b1) {
  asm volatile(
      "{\n\t.reg .f32 z0, z1;\n\t"
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, z0, z1}, "
      "{%2, %4, %3, %4}, {%5, %6}, {%0, %1, %7, %7};\n\t}"
      : "+f"(d[0]), "+f"(d[1])
      : "r"(a0), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
}

// Bytes {a.b[j], b.b[j], a.b[j+1], b.b[j+1]} for j = 0 (even m-tile) or 2.
__device__ __forceinline__ uint32_t interleave2(uint32_t a, uint32_t b, int j) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(j ? 0x7362u : 0x5140u));
  return r;
}

// Byte offset, inside a unit's K or V tile, of the 16-byte chunk `chunk`
// (8 dims) of key row `tok`: 64-dim box, row, 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int tok, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (kUnit * 128) + tok * 128 +
                               (((chunk & 7) ^ (tok & 7)) << 4));
}

// HALF: the CTA's rows are 8 or fewer (a single-token decode of up to 8
// heads per KV head): rows 8..15 of the m16 tile are not kept at all.
// CTAs per SM: the fp8 half-tile variant (34 KB of shared memory) runs 4
// within 128 registers (a few spilled bytes; 0.745 vs 0.711 of HBM with 3);
// the 16-bit variants are held to 3 by their shared memory (71 KB), the fp8
// 16-row variant by its registers.
template <bool KV8, bool HALF>
constexpr int kDecodeCtasPerSm = (KV8 && HALF) ? 4 : 3;
template <class T, int D, bool KV8, bool HALF>
__global__ void __launch_bounds__(kThreads, kDecodeCtasPerSm<KV8, HALF>)
decode_kernel(const Args a, const __grid_constant__ CUtensorMap tmap) {
  using L = Lay<D, KV8>;
  using MT = std::conditional_t<KV8, FP16, T>;  // MMA operand type (and P)
  constexpr int NR = HALF ? 1 : 2;              // row halves a lane keeps (g, g + 8)
  constexpr int KS = D / 16;  // k-steps of q.k
  constexpr int NT = D / 8;   // n-tiles of p.V
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / a.row_groups, rg = blockIdx.y % a.row_groups;
  const int b = blockIdx.z;
  const int H = a.H, q = a.q, QPK = a.QPK;
  // launched as a dependent of the stream's previous kernel: its outputs (the
  // cache writes, the query) are read only past this wait; the split combine
  // may be scheduled as soon as every CTA of this grid is running
  grid_dependency_wait();
  grid_launch_dependents();
  const Span sp = span_of(a, b, split == 0 && blockIdx.y == 0 && threadIdx.x == 0);

  // this lane's two rows of the m16 tile: g and g + 8
  const int g = lane >> 2, tq = lane & 3;
  int R[2], orow[2], pos[2], lo[2];
  bool valid[2];
  float slope[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    R[x] = rg * kRows + g + 8 * x;
    valid[x] = R[x] < a.rows && x < NR;
    const int t = valid[x] ? R[x] / QPK : 0, h = valid[x] ? R[x] % QPK : 0;
    const int head = kvh * QPK + h;
    orow[x] = (b * q + t) * H + head;  // output row (token, head)
    pos[x] = sp.L - q + t;
    lo[x] = a.window > 0 ? max(0, pos[x] - a.window + 1) : 0;
    slope[x] = (a.alibi && valid[x]) ? __ldg(a.alibi + head) * kLog2e : 0.f;
  }

  if (sp.L == 0 || sp.nunits == 0) {
    // padding (or a reported bad length): zero rows; a rank holding no
    // visible key: the empty partial (o = 0, m = -inf, l = 0)
    if (split == 0 && warp == 0) {
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (valid[x]) {
          const int64_t hh = orow[x];
          if (a.res_o) {
            for (int d = tq; d < D; d += 4) a.res_o[hh * D + d] = 0.f;
            if (tq == 0) {
              a.res_ml[hh * 2] = -INFINITY;
              a.res_ml[hh * 2 + 1] = 0.f;
            }
          } else {
            uint16_t *o16 = static_cast<uint16_t *>(a.out);
            for (int d = tq; d < D; d += 4) o16[hh * D + d] = 0;
          }
        }
    }
    return;
  }
  const int u_begin = sp.first_unit + split * a.split_units;
  const int u_end = min(u_begin + a.split_units, sp.first_unit + sp.nunits);
  if (split >= sp.nsplit || u_begin >= u_end) return;
  const int nu = u_end - u_begin;

  uint8_t *tiles = smem;
  int32_t *coord = reinterpret_cast<int32_t *>(smem + L::TILES);
  uint64_t *bars = reinterpret_cast<uint64_t *>(
      smem + L::TILES + ((a.split_units * 4 + 15) / 16) * 16);

  if (threadIdx.x == 0) prefetch_tensormap(&tmap);
  // cache row coordinate of each unit of the split, range-checked once
  const int32_t *trow = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
  for (int k = threadIdx.x; k < nu; k += kThreads) {
    const int p0 = (u_begin + k) * kUnit;
    const int lb = p0 / a.BS;
    int pb = __ldg(trow + lb);
    if (pb < 0 || pb >= a.num_blocks) {
      record_error(PKV_ERR_BOUNDS, static_cast<int64_t>(b) * a.max_blocks_per_seq + lb);
      pb = 0;
    }
    coord[k] = pb * a.BS + p0 % a.BS;
  }
  if constexpr (!KV8)  // the zero V tile (16-bit cache only)
    for (int i = threadIdx.x; i < L::V16 / 16; i += kThreads)
      reinterpret_cast<uint4 *>(tiles + L::ZERO)[i] = make_uint4(0u, 0u, 0u, 0u);
  uint64_t *wbar = bars + warp * L::NST;
  if (lane == 0) {
    for (int st = 0; st < L::NST; ++st) mbar_init(&wbar[st], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int my_count = nu > warp ? (nu - warp + kWarps - 1) / kWarps : 0;
  uint8_t *wt = tiles + warp * L::NST * L::STAGE;
  auto issue = [&](int k) {
    const int st = k % L::NST;
    const int c = coord[warp + k * kWarps];
    mbar_arrive_expect_tx(&wbar[st], 2u * L::TILE);
    uint8_t *kt = wt + st * L::STAGE;
    if constexpr (KV8) {  // one box of 16 rows x D codes each
      tma_load_4d(kt, &tmap, &wbar[st], 0, kvh, c, 0);
      tma_load_4d(kt + L::TILE, &tmap, &wbar[st], 0, kvh, c, 1);
    } else {
#pragma unroll
      for (int r = 0; r < D / 64; ++r) {
        tma_load_4d(kt + r * L::BOX, &tmap, &wbar[st], 64 * r, kvh, c, 0);
        tma_load_4d(kt + L::TILE + r * L::BOX, &tmap, &wbar[st], 64 * r, kvh, c, 1);
      }
    }
  };
  int issued = 0;
  if (lane == 0)
    for (; issued < min(L::NST, my_count); ++issued) issue(issued);

  // ---- Q fragments (A operand, row-major 16 x 16 per k-step) ---------------
  uint32_t qa[KS][4];
  float sl2 = a.scale_log2;
  // fp8 cache, four rows or fewer (a single-token decode of up to 4 heads per
  // KV head): rows 4..7 of the m16 tile carry the lo query terms of rows
  // 0..3, so one product per k-step gives both terms (summed across lanes).
  const bool fold = KV8 && HALF && a.rows <= 4;
  if constexpr (KV8) {
    // E4M3 terms: qa[s] = hi, qa[KS8 + s] = lo of k-step s (32 positions):
    // positions 4tq .. 4tq+3 -> dims tq * D/4 + 8s + 0..3, positions
    // 16 + 4tq .. -> dims tq * D/4 + 8s + 4..7 (eight consecutive elements)
    constexpr int KS8 = D / 32;
    const int srow = fold ? (g & 3) : g;  // the row whose query this lane's row 0 holds
    const bool lo_lane = fold && g >= 4;
    const bool src_valid = fold ? rg * kRows + srow < a.rows : valid[0];
    const int64_t src_orow = fold ? static_cast<int64_t>(b * q + (rg * kRows + srow) / QPK) * H +
                                        kvh * QPK + (rg * kRows + srow) % QPK
                                  : orow[0];
    auto qchunk = [&](int x, int s) -> uint4 {  // this lane's dims tq * D/4 + 8s .. + 7 of row x
      const int64_t r = x == 0 ? src_orow : orow[x];
      const bool v = x == 0 ? src_valid : valid[x];
      const uint4 *qp = reinterpret_cast<const uint4 *>(a.query) + (r * D + tq * (D / 4)) / 8;
      return v ? __ldg(qp + s) : make_uint4(0u, 0u, 0u, 0u);
    };
    uint32_t am = 0;  // largest |q| bit pattern (fp32)
#pragma unroll
    for (int x = 0; x < NR; ++x)
#pragma unroll
      for (int s = 0; s < KS8; ++s) {
        const uint4 u = qchunk(x, s);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = T::to_f2(word_of(u, k));
          am = max(am, max(__float_as_uint(fabsf(f.x)), __float_as_uint(fabsf(f.y))));
        }
      }
    // every warp holds the whole row group, so a warp's max is the group's
    am = __reduce_max_sync(0xffffffffu, am);
    const int E = static_cast<int>(am >> 23);
    // largest |q| * 2^-e in [2^7, 2^8): hi and lo inside E4M3's range
    const int e = E == 0 ? 0 : min(64, max(-64, E - 134));
    const float mul = __int_as_float((127 - e) << 23);
    sl2 *= __int_as_float((127 + e) << 23);
#pragma unroll
    for (int s = 0; s < KS; ++s)
#pragma unroll
      for (int c = 0; c < 4; ++c) qa[s][c] = 0u;
#pragma unroll
    for (int x = 0; x < NR; ++x)
#pragma unroll
      for (int s = 0; s < KS8; ++s) {
        const uint4 u = qchunk(x, s);
        float v[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = T::to_f2(word_of(u, k));
          v[2 * k] = f.x * mul;
          v[2 * k + 1] = f.y * mul;
        }
        split_e4m3x4(v[0], v[1], v[2], v[3], qa[s][x], qa[KS8 + s][x]);
        split_e4m3x4(v[4], v[5], v[6], v[7], qa[s][2 + x], qa[KS8 + s][2 + x]);
        if (x == 0 && lo_lane) {  // rows 4..7 hold the lo terms
          qa[s][0] = qa[KS8 + s][0];
          qa[s][2] = qa[KS8 + s][2];
        }
      }
  } else {
    const uint32_t *q0 = reinterpret_cast<const uint32_t *>(a.query) +
                         (static_cast<int64_t>(orow[0]) * D) / 2;
    const uint32_t *q1 = reinterpret_cast<const uint32_t *>(a.query) +
                         (static_cast<int64_t>(orow[1]) * D) / 2;
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      qa[s][0] = valid[0] ? __ldg(q0 + 8 * s + tq) : 0u;
      qa[s][1] = valid[1] ? __ldg(q1 + 8 * s + tq) : 0u;
      qa[s][2] = valid[0] ? __ldg(q0 + 8 * s + 4 + tq) : 0u;
      qa[s][3] = valid[1] ? __ldg(q1 + 8 * s + 4 + tq) : 0u;
    }
  }

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[NT][2 * NR];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int c = 0; c < 2 * NR; ++c) o[n][c] = 0.f;
  // fp8 cache: the same registers as O^T tiles: ot[mt][nt][c] holds dims
  // dm(mt) + (c >> 1) (dm(mt) = 16g + 2mt for D = 128, 8g + 2mt for D = 64)
  // of query rows 8nt + 2tq + (c & 1)
  float(&ot)[D / 16][NR][4] = *reinterpret_cast<float(*)[D / 16][NR][4]>(&o[0][0]);
  // keys every row of the CTA sees: no masking needed on a unit inside them
  const int pos_min = sp.L - q;  // token 0
  const int lo_max = a.window > 0 ? max(0, sp.L - a.window) : 0;  // last token's window start
  const bool has_alibi = a.alibi != nullptr;
  const int RW = a.dcp_world;  // local key k sits at position k * RW + dcp_rank
  const float tq2 = static_cast<float>(2 * tq * RW);

  // ldmatrix row addresses: lane -> (matrix mi, row rr)
  const int mi = lane >> 3, rr = lane & 7;
  const int k_tok = (mi >> 1) * 8 + rr, k_half = mi & 1;  // K: tokens x dim halves
  const int v_tok = (mi & 1) * 8 + rr, v_half = mi >> 1;  // V^T: token halves x dims
  bool ok = true;
  int consumed = 0;

  for (int k = 0; k < my_count; ++k) {
    const int st = k % L::NST;
    const bool got = mbar_wait_bounded(&wbar[st], (k / L::NST) & 1, b);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    consumed = k + 1;
    const uint32_t kt = smem_u32(wt + st * L::STAGE);
    uint32_t vt = kt + L::TILE;
    // position of the unit's key 0 (its keys are R positions apart)
    const int j0 = (u_begin + warp + k * kWarps) * kUnit * RW + a.dcp_rank;

    // ---- S = Q K^T: two n-tiles of 8 keys ---------------------------------
    // Even and odd k-steps accumulate apart (summed below): four independent
    // MMA chains of KS / 2 instead of two of KS, for the latency.
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float sc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    // product of k-step s into n-tile n (the top half only, with HALF)
    auto mma_s = [&](int n, int s, const uint32_t (&qs)[4], uint32_t b0, uint32_t b1) {
      float(&acc)[4] = (s & 1) ? sc2[n] : sc[n];
      if constexpr (HALF) {
        float d2[2] = {acc[0], acc[1]};
        mma16816_top<MT>(d2, qs[0], qs[2], b0, b1);
        acc[0] = d2[0];
        acc[1] = d2[1];
      } else {
        mma16816<MT>(acc, qs, b0, b1);
      }
    };
    if constexpr (KV8) {
      // keys g and g + 8: this lane's D/4 codes of each (its chunks of the
      // swizzled rows), straight into the E4M3 products, hi then lo terms
      constexpr int KS8 = D / 32, KC = D / 64;
      const uint8_t *kc = wt + st * L::STAGE;
      uint4 kk[2][KC];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int c = 0; c < KC; ++c)
          kk[n][c] = *reinterpret_cast<const uint4 *>(kc + swz8<D>(g + 8 * n, tq * KC + c));
#pragma unroll
      for (int s = 0; s < KS8; ++s)
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const uint32_t b0 = word_of(kk[n][(2 * s) / 4], (2 * s) % 4);
          const uint32_t b1 = word_of(kk[n][(2 * s + 1) / 4], (2 * s + 1) % 4);
          if constexpr (HALF) {
            if (fold) {  // both terms in one product: even / odd k-steps apart
              float(&acc)[4] = (s & 1) ? sc2[n] : sc[n];
              float d2[2] = {acc[0], acc[1]};
              mma16832_e4m3_top(d2, qa[s][0], qa[s][2], b0, b1);
              acc[0] = d2[0];
              acc[1] = d2[1];
            } else {
              float d2[2] = {sc[n][0], sc[n][1]};
              mma16832_e4m3_top(d2, qa[s][0], qa[s][2], b0, b1);
              sc[n][0] = d2[0];
              sc[n][1] = d2[1];
              float e2[2] = {sc2[n][0], sc2[n][1]};
              mma16832_e4m3_top(e2, qa[KS8 + s][0], qa[KS8 + s][2], b0, b1);
              sc2[n][0] = e2[0];
              sc2[n][1] = e2[1];
            }
          } else {
            mma16832_e4m3(sc[n], qa[s], b0, b1);
            mma16832_e4m3(sc2[n], qa[KS8 + s], b0, b1);
          }
        }
    } else {
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        uint32_t kb[4];
        ldsm_x4(kt + swz(k_tok, 2 * s + k_half), kb);
        mma_s(0, s, qa[s], kb[0], kb[1]);
        mma_s(1, s, qa[s], kb[2], kb[3]);
      }
    }
    // ---- scores in the log2 domain, per-row masks --------------------------
    // sc[n][e] : row g (e < 2) or g + 8 (e >= 2), key j0 + 8n + 2tq + (e & 1)
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int c = 0; c < 2 * NR; ++c) sc[n][c] += sc2[n][c];
    if constexpr (KV8 && HALF) {
      if (fold) {  // row g + 4 holds row g's lo-term product (lane + 16)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int c = 0; c < 2; ++c) sc[n][c] += __shfl_xor_sync(0xffffffffu, sc[n][c], 16);
      }
    }
    // A unit inside [lo_max, pos_min] needs no mask (rows past a.rows hold
    // zero queries; their results are never stored).
    const bool interior = j0 >= lo_max && j0 + (kUnit - 1) * RW <= pos_min;
    float x[2][4];  // [row][n * 2 + (e & 1)]
    bool grow = false;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float rel = static_cast<float>(j0 - pos[r]) + tq2;  // key j0 + 2tq minus i
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float v = sc[n][2 * r + c] * sl2;
          if (has_alibi) v = fmaf(slope[r], rel + static_cast<float>((8 * n + c) * RW), v);
          if (!interior) {
            const int j = j0 + (8 * n + 2 * tq + c) * RW;
            if (!valid[r] || j < lo[r] || j > pos[r]) v = -INFINITY;
          }
          x[r][n * 2 + c] = v;
          grow |= v > m[r] + kLazy;
        }
    }
    if (__any_sync(0xffffffffu, grow)) {
      // move the references to the true row maxima (4 lanes hold a row)
      float al[2] = {1.f, 1.f};
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float mx = fmaxf(fmaxf(x[r][0], x[r][1]), fmaxf(x[r][2], x[r][3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m[r], mx);
        if (mn > m[r]) {
          const float alpha = m[r] == -INFINITY ? 0.f : fast_exp2(m[r] - mn);
          m[r] = mn;
          l[r] *= alpha;
          al[r] = alpha;
          if constexpr (!KV8) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              o[n][2 * r] *= alpha;
              o[n][2 * r + 1] *= alpha;
            }
          }
        }
      }
      if constexpr (KV8) {
        // O^T columns are query rows 8nt + 2tq, + 1, owned by lanes 8tq, 8tq + 4
#pragma unroll
        for (int nt = 0; nt < NR; ++nt) {
          const float a0 = __shfl_sync(0xffffffffu, al[nt], 8 * tq);
          const float a1 = __shfl_sync(0xffffffffu, al[nt], 8 * tq + 4);
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            ot[mt][nt][0] *= a0;
            ot[mt][nt][1] *= a1;
            ot[mt][nt][2] *= a0;
            ot[mt][nt][3] *= a1;
          }
        }
      }
    }
    // ---- P (A operand of P V): rows g / g + 8, keys 2tq.. and 8 + 2tq.. -----
    uint32_t pa[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float mr = m[r] == -INFINITY ? 0.f : m[r];
      float p[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) p[c] = fast_exp2(x[r][c] - mr);
      l[r] += (p[0] + p[1]) + (p[2] + p[3]);
      pa[r] = MT::from_f2(p[0], p[1]);      // keys 2tq, 2tq + 1
      pa[2 + r] = MT::from_f2(p[2], p[3]);  // keys 8 + 2tq, 9 + 2tq
    }
    // Slots past the rank's last token in its last cache block hold whatever
    // the cache holds there, possibly non-finite: their P is exactly 0, but
    // 0 * NaN is NaN, so V rows of such slots are read as zeros (16-bit
    // cache: the lanes whose ldmatrix row is such a slot read the zero tile;
    // fp8: the codes of such rows are replaced by zeros).  Stale K rows need
    // nothing: their scores are masked to -inf.
    if constexpr (KV8) {
      // ---- O^T += V^T P^T: m-tiles of 16 dims, P fragments as the B operand
      constexpr int VW = D / 32;  // words of this lane's chunk of a key row
      const uint8_t *vc = wt + st * L::STAGE + L::TILE;
      const bool tail = j0 + (kUnit - 1) * RW >= pos_min + q;
      uint32_t vw[4][VW];  // keys 2tq, 2tq + 1, 2tq + 8, 2tq + 9
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int kr = 2 * tq + (kk & 1) + 8 * (kk >> 1);
        if constexpr (D == 128) {
          const uint4 u = *reinterpret_cast<const uint4 *>(vc + swz8<D>(kr, g));
          vw[kk][0] = u.x;
          vw[kk][1] = u.y;
          vw[kk][2] = u.z;
          vw[kk][3] = u.w;
        } else {
          const uint2 u =
              *reinterpret_cast<const uint2 *>(vc + swz8<D>(kr, g >> 1) + 8 * (g & 1));
          vw[kk][0] = u.x;
          vw[kk][1] = u.y;
        }
        if (tail && j0 + kr * RW >= pos_min + q) {
#pragma unroll
          for (int w = 0; w < VW; ++w) vw[kk][w] = 0u;
        }
      }
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        // A rows g / g + 8 = dims dm(mt) / dm(mt) + 1: bytes 2mt, 2mt + 1 of
        // the lane's chunk, keys paired as the fragment wants them
        const int w = mt >> 1, j = (mt & 1) * 2;
        const uint2 h01 = e4m3x4_to_h4(interleave2(vw[0][w], vw[1][w], j));
        const uint2 h89 = e4m3x4_to_h4(interleave2(vw[2][w], vw[3][w], j));
        const uint32_t av[4] = {h01.x, h01.y, h89.x, h89.y};
        mma16816<FP16>(ot[mt][0], av, pa[0], pa[2]);
        if constexpr (!HALF) mma16816<FP16>(ot[mt][1], av, pa[1], pa[3]);
      }
    } else {
      if (j0 + v_tok * RW >= pos_min + q) vt = smem_u32(tiles + L::ZERO);
      // ---- O += P V: n-tiles of 8 dims, two per ldmatrix -------------------
#pragma unroll
      for (int n2 = 0; n2 < NT / 2; ++n2) {
        uint32_t vb[4];
        ldsm_x4_t(vt + swz(v_tok, 2 * n2 + v_half), vb);
        if constexpr (HALF) {
          mma16816_top<MT>(o[2 * n2], pa[0], pa[2], vb[0], vb[1]);
          mma16816_top<MT>(o[2 * n2 + 1], pa[0], pa[2], vb[2], vb[3]);
        } else {
          mma16816<MT>(o[2 * n2], pa, vb[0], vb[1]);
          mma16816<MT>(o[2 * n2 + 1], pa, vb[2], vb[3]);
        }
      }
    }
    __syncwarp();  // every lane has read the stage: refill it
    if (lane == 0 && issued < my_count) {
      issue(issued);
      ++issued;
    }
    __syncwarp();
  }
  issued = __shfl_sync(0xffffffffu, issued, 0);
  if (!ok) {  // drain this warp's copies still in flight, bounded
    for (int k = consumed; k < issued; ++k) mbar_wait_bounded(&wbar[k % L::NST], (k / L::NST) & 1, b);
  }

  // ---- merge the 4 warps' (m, l, O) ----------------------------------------
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  __syncthreads();  // all TMA traffic has landed; the tile area is reusable
  float *sM = reinterpret_cast<float *>(smem);  // [warp][row]
  float *sL = sM + kWarps * kRows;               // [warp][row]
  float *sO = sL + kWarps * kRows;               // [warp][row][D]
  if (tq == 0) {
    sM[warp * kRows + g] = ok ? m[0] : -INFINITY;
    sM[warp * kRows + g + 8] = ok ? m[1] : -INFINITY;
    sL[warp * kRows + g] = ok ? l[0] : 0.f;
    sL[warp * kRows + g + 8] = ok ? l[1] : 0.f;
  }
  if constexpr (KV8) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int nt = 0; nt < NR; ++nt) {
        float *r0 = sO + (warp * kRows + 8 * nt + 2 * tq) * D + (D == 128 ? 16 : 8) * g + 2 * mt;
        r0[0] = ot[mt][nt][0];
        r0[D] = ot[mt][nt][1];
        r0[1] = ot[mt][nt][2];
        r0[D + 1] = ot[mt][nt][3];
      }
  } else {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      float *r0 = sO + (warp * kRows + g) * D + 8 * n + 2 * tq;
      r0[0] = o[n][0];
      r0[1] = o[n][1];
      if constexpr (!HALF) {
        r0[8 * D] = o[n][2];
        r0[8 * D + 1] = o[n][3];
      }
    }
  }
  __syncthreads();
  const bool single = sp.nsplit == 1;
  for (int idx = threadIdx.x; idx < kRows * D; idx += kThreads) {
    const int r = idx / D, d = idx % D;
    const int Rr = rg * kRows + r;
    if (Rr >= a.rows) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sM[w * kRows + r]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float e = fast_exp2(sM[w * kRows + r] - M);
        num = fmaf(e, sO[(w * kRows + r) * D + d], num);
        den = fmaf(e, sL[w * kRows + r], den);
      }
    }
    const float val = den > 0.f ? num / den * a.v_scale : 0.f;
    const int t = Rr / QPK, h = Rr % QPK;
    const int64_t hh = static_cast<int64_t>(b * q + t) * H + kvh * QPK + h;
    if (single && a.res_o) {  // this rank's share, whole: its (o, m, l)
      a.res_o[hh * D + d] = val;
      if (d == 0) {
        a.res_ml[hh * 2] = M;
        a.res_ml[hh * 2 + 1] = den;
      }
    } else if (single) {
      uint16_t *o16 = static_cast<uint16_t *>(a.out);
      o16[hh * D + d] = static_cast<uint16_t>(T::from_f2(val, 0.f) & 0xffffu);
    } else {
      const int64_t slot = hh * a.max_splits + split;
      a.part_o[slot * D + d] = val;
      if (d == 0) {
        a.part_ml[slot * 2] = M;
        a.part_ml[slot * 2 + 1] = den;
      }
    }
  }
}

// Merge of a row's split partials (a3): one warp per (decode token row,
// query head), four heads per CTA; lane l owns dims l * D/32 ...
template <class T, int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const Args a) {
  constexpr int EPL = D / 32;  // dims per lane
  grid_dependency_wait();  // the split kernel's partials are complete and visible
  const int row = blockIdx.x;  // row = b * q + t
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 4 + warp;
  const Span sp = span_of(a, row / a.q, false);
  if (h >= a.H || sp.L == 0 || sp.nsplit <= 1) return;  // else written by the split kernel
  const int64_t hh = static_cast<int64_t>(row) * a.H + h;
  const float *ml = a.part_ml + hh * a.max_splits * 2;
  float M = -INFINITY;
  for (int s = lane; s < sp.nsplit; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float num[EPL], den = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) num[e] = 0.f;
  if (M != -INFINITY) {
    const float *po = a.part_o + hh * a.max_splits * D + lane * EPL;
    // four splits' loads in flight at a time (the partials come from L2)
    constexpr int G = 4;
    for (int s0 = 0; s0 < sp.nsplit; s0 += G) {
      float mm[G], ll[G], v[G][EPL];
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const int s = min(s0 + i, sp.nsplit - 1);
        mm[i] = ml[2 * s];
        ll[i] = ml[2 * s + 1];
        if constexpr (EPL == 4) {
          const float4 t = *reinterpret_cast<const float4 *>(po + static_cast<int64_t>(s) * D);
          v[i][0] = t.x; v[i][1] = t.y; v[i][2] = t.z; v[i][3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2 *>(po + static_cast<int64_t>(s) * D);
          v[i][0] = t.x; v[i][1] = t.y;
        }
      }
#pragma unroll
      for (int i = 0; i < G; ++i) {
        if (s0 + i >= sp.nsplit) break;
        const float w = fast_exp2(mm[i] - M) * ll[i];
#pragma unroll
        for (int e = 0; e < EPL; ++e) num[e] = fmaf(w, v[i][e], num[e]);
        den += w;
      }
    }
  }
  float val[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) val[e] = den > 0.f ? num[e] / den : 0.f;
  if (a.res_o) {  // this rank's share: its merged (o, m, l)
    float *ro = a.res_o + hh * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) ro[e] = val[e];
    if (lane == 0) {
      a.res_ml[hh * 2] = M;
      a.res_ml[hh * 2 + 1] = den;
    }
    return;
  }
  uint32_t *o32 = reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(a.out) + hh * D + lane * EPL);
#pragma unroll
  for (int e = 0; e < EPL; e += 2) o32[e / 2] = T::from_f2(val[e], val[e + 1]);
}

// Decode context parallelism: merge the ranks' (o, m, l) of each (row, head)
// (a3 across ranks).  parts_o [P][rows * H][D], parts_ml [P][rows * H][2],
// rank-major as an all-gather lays them out.  One warp per (row, head), four
// heads per CTA, lane l owning dims l * D/32 ...
template <class T, int D>
__global__ void __launch_bounds__(128)
dcp_combine_kernel(void *out, const float *parts_o, const float *parts_ml, int num_parts,
                   int64_t rows_heads, int H) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 4 + warp;
  if (h >= H) return;
  const int64_t hh = static_cast<int64_t>(blockIdx.x) * H + h;
  float M = -INFINITY;
  for (int p = lane; p < num_parts; p += 32) M = fmaxf(M, parts_ml[(p * rows_heads + hh) * 2]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float num[EPL], den = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) num[e] = 0.f;
  if (M != -INFINITY) {
    for (int p = 0; p < num_parts; ++p) {
      const float l = parts_ml[(p * rows_heads + hh) * 2 + 1];
      if (l <= 0.f) continue;  // the rank holds no visible key
      const float w = fast_exp2(parts_ml[(p * rows_heads + hh) * 2] - M) * l;
      const float *po = parts_o + (p * rows_heads + hh) * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) num[e] = fmaf(w, po[e], num[e]);
      den += w;
    }
  }
  uint32_t *o32 = reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(out) + hh * D + lane * EPL);
#pragma unroll
  for (int e = 0; e < EPL; e += 2)
    o32[e / 2] = T::from_f2(den > 0.f ? num[e] / den : 0.f, den > 0.f ? num[e + 1] / den : 0.f);
}

template <class T, int D, bool KV8>
static cudaError_t launch_typed(const Args &a, const CUtensorMap &tmap, int KVH, int num_seqs,
                                cudaStream_t stream) {
  const size_t table = ((a.split_units * 4 + 15) / 16) * 16;
  const size_t smem = 1024 + Lay<D, KV8>::TILES + table + kWarps * Lay<D, KV8>::NST * 8;
  auto kern = a.rows <= kRows / 2 ? decode_kernel<T, D, KV8, true> : decode_kernel<T, D, KV8, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // both kernels are programmatic dependents of the kernel before them in the
  // stream (each waits for it before its first global read), so their launch
  // overlaps the previous kernel's tail
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.max_splits, KVH * a.row_groups, num_seqs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a, tmap);
  if (e != cudaSuccess || a.max_splits <= 1) return e;
  cfg.gridDim = dim3(num_seqs * a.q, (a.H + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<T, D>, a);
}

}  // namespace dec

DecodePlan plan_decode(int num_seqs, int query_len, int max_seq_len, const Geometry &g, int sms,
                       int dcp_world) {
  DecodePlan p{};
  const int U = dec::kUnit;
  // keys (of this rank) the batch's widest row set can see
  int eff = std::max(max_seq_len, 1);
  if (g.window > 0 && g.window + query_len - 1 < eff) eff = g.window + query_len - 1;
  eff = (eff + dcp_world - 1) / dcp_world + (dcp_world > 1 ? 1 : 0);
  const int units = (eff + U - 1) / U + 1;  // a window start can straddle a unit
  p.row_groups = (query_len * g.QPK + dec::kRows - 1) / dec::kRows;
  const int64_t items = static_cast<int64_t>(num_seqs) * g.KVH * p.row_groups;
  // Splits of up to 256 units (4096 keys): every split writes fp32 partials of
  // all its q * QPK rows, so short splits cost real HBM traffic; shrink them
  // only while the grid would leave SMs idle.  (Measured on 128 sequences x 4
  // tokens, 512..4096 keys: 0.71 / 0.82 / 0.85 / 0.876 of HBM with 32 / 64 /
  // 128 / 256; 256 sequences x 1 token: 0.970 / 0.979 with 128 / 256, where
  // 256 leaves one split per sequence and no combine pass.)
  int split_units = 256;
  while (split_units > 8 && items * ((units + split_units - 1) / split_units) < 8LL * sms)
    split_units /= 2;
  if (units <= 2 * split_units) split_units = units;  // short: one split
  p.split_units = split_units;
  p.max_splits = (units + split_units - 1) / split_units;
  if (p.max_splits > 1) {
    const size_t rows = static_cast<size_t>(num_seqs) * query_len * g.H * p.max_splits;
    const size_t o_bytes = ((rows * g.D * 4 + 255) / 256) * 256;
    const size_t ml_bytes = ((rows * 2 * 4 + 255) / 256) * 256;
    p.workspace_bytes = o_bytes + ml_bytes;
  }
  return p;
}

cudaError_t launch_decode(void *out, const void *query, int num_seqs, int query_len,
                          const void *kv_cache, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *seq_lens, const Geometry &g,
                          const DecodePlan &plan, void *workspace, cudaStream_t stream,
                          const DcpShare &dcp) {
  CUtensorMap tmap;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.D), static_cast<cuuint64_t>(g.KVH),
                              static_cast<cuuint64_t>(g.num_blocks * g.BS), 2};
  const cuuint64_t eb = static_cast<cuuint64_t>(g.elem_bytes);
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.D) * eb,
                                 static_cast<cuuint64_t>(g.row_elems) * eb,
                                 static_cast<cuuint64_t>(g.num_blocks * g.block_elems) * eb};
  // 16-bit cache: 64-dim boxes, 128-byte swizzle (ldmatrix reads them);
  // fp8 cache: one box of D codes per row, swizzled by its row length
  const cuuint32_t box[4] = {g.fp8 ? static_cast<cuuint32_t>(g.D) : 64u, 1,
                             static_cast<cuuint32_t>(dec::kUnit), 1};
  const bool bf = g.dtype == PKV_BF16;
  const CUtensorMapDataType dt =
      g.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
            : (bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  const CUtensorMapSwizzle swz = !g.fp8 || g.D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                     : CU_TENSOR_MAP_SWIZZLE_64B;
  if (encode_tensor_map(&tmap, dt, 4, const_cast<void *>(kv_cache), dims, strides, box, swz) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  dec::Args a{};
  a.out = out;
  a.query = static_cast<const uint16_t *>(query);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.alibi = g.alibi;
  if (plan.max_splits > 1) {
    const size_t rows = static_cast<size_t>(num_seqs) * query_len * g.H * plan.max_splits;
    const size_t o_bytes = ((rows * g.D * 4 + 255) / 256) * 256;
    a.part_o = static_cast<float *>(workspace);
    a.part_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + o_bytes);
  }
  a.num_blocks = g.num_blocks;
  a.num_seqs = num_seqs;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.H = g.H;
  a.QPK = g.QPK;
  a.q = query_len;
  a.rows = query_len * g.QPK;
  a.row_groups = plan.row_groups;
  a.BS = g.BS;
  a.window = g.window;
  a.split_units = plan.split_units;
  a.max_splits = plan.max_splits;
  a.scale_log2 = g.scale * kLog2e * g.k_scale;
  a.v_scale = g.v_scale;
  a.dcp_world = dcp.world;
  a.dcp_rank = dcp.rank;
  a.res_o = dcp.res_o;
  a.res_ml = dcp.res_ml;
#define PKV_MT(TT, DD)                                                             \
  if (g.D == DD)                                                                   \
    return g.fp8 ? dec::launch_typed<TT, DD, true>(a, tmap, g.KVH, num_seqs, stream) \
                 : dec::launch_typed<TT, DD, false>(a, tmap, g.KVH, num_seqs, stream);
  if (bf) {
    PKV_MT(BF16, 128) PKV_MT(BF16, 64)
  } else {
    PKV_MT(FP16, 128) PKV_MT(FP16, 64)
  }
#undef PKV_MT
  return cudaErrorInvalidValue;
}


cudaError_t launch_dcp_combine(void *out, const float *parts_o, const float *parts_ml,
                              int num_parts, int64_t num_rows, const Geometry &g,
                              cudaStream_t stream) {
  if (num_rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(num_rows), static_cast<unsigned>((g.H + 3) / 4));
  const int64_t rh = num_rows * g.H;
  const bool bf = g.dtype == PKV_BF16;
  if (g.D == 128) {
    if (bf) dec::dcp_combine_kernel<BF16, 128><<<grid, 128, 0, stream>>>(out, parts_o, parts_ml, num_parts, rh, g.H);
    else dec::dcp_combine_kernel<FP16, 128><<<grid, 128, 0, stream>>>(out, parts_o, parts_ml, num_parts, rh, g.H);
  } else if (g.D == 64) {
    if (bf) dec::dcp_combine_kernel<BF16, 64><<<grid, 128, 0, stream>>>(out, parts_o, parts_ml, num_parts, rh, g.H);
    else dec::dcp_combine_kernel<FP16, 64><<<grid, 128, 0, stream>>>(out, parts_o, parts_ml, num_parts, rh, g.H);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Static decode scratch for callers that cannot allocate device memory.
//
// The split partials of paged_attn_decode_noalloc live in this file-scope
// array instead of a caller workspace.  The array belongs to the module, so
// every GPU that loads this library holds it until the process exits.  In
// host code its name is only a host-side stand-in: the device address must be
// looked up (once per device, with that device current) and passed to the
// kernels.  All calls share the array and it keeps the last call's contents;
// nothing in it has to start at zero, because the combine pass only reads
// partials the split pass of the same call has just written.  Calls whose
// work overlaps on the GPU (different streams, or before the previous call
// has finished) race on it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_DECODE_STATIC_SCRATCH_BYTES];

static void *g_scratch_addr[64];
static bool g_scratch_known[64];
static std::mutex g_scratch_mu;

cudaError_t static_decode_scratch(int dev, void **ptr, size_t *bytes) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return e;
  // the symbol's address is looked up with its own device current
  if (dev < 0 || dev >= 64 || dev != cur) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_known[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
    g_scratch_known[dev] = true;
  }
  *ptr = g_scratch_addr[dev];
  *bytes = sizeof(g_decode_scratch);
  return cudaSuccess;
}

cudaError_t read_device_error_decode(unsigned long long *out) {
  return read_and_clear_unit_error(out);
}

}  // namespace pkv
