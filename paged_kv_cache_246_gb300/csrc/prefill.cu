// Varlen causal prefill over the paged cache, with or without a cached
// context (chunked prefill), on the 5th-generation tensor core.
//
// What is computed (xformers.py XFormersImpl.forward -> forward_prefix and
// _run_memory_efficient_xformers_forward; cpu_attn flash_attn_varlen_func):
// sequence b has L_b = cu_k[b+1] - cu_k[b] tokens of which the last
// q_b = cu_q[b+1] - cu_q[b] are query rows; row t sits at position
// i = (L_b - q_b) + t and attends to keys lo(i) <= j <= i of its sequence
// (every key 0 <= j < L_b for encoder attention, non_causal), all read
// through the block table:
//     s_j = scale * q.k_j + slope_h * (j - i),   out = softmax(s) . V.
//
// Design: CTA = two 128-row query tiles sharing every K/V tile: two query
// heads of one KV group on the same rows when the group has an even number
// of heads (grouped-query reuse), else one head on two consecutive row tiles.
// 12 warps:
//   warp 0      TMA producer: the two Q tiles once; per 128-key tile the K
//               and V rows of the KV head, one box (block_size rows x 64 dims,
//               128-byte swizzle) per cache block and 64-dim half, straight
//               from the paged cache.  Blocks outside the visible range are
//               loaded from an out-of-range coordinate, which the TMA unit
//               zero-fills.  K and V have 2 stages each, each freed by its own
//               barrier (a K stage when its QK products are done, a V stage
//               when its PV products are done), and the next tile's
//               block-table entries are fetched one tile ahead, so copies
//               start a full tile before the tensor core needs them.
//   warp 1      MMA issuer (one thread), in the order
//                 QK_A(0) QK_B(0) | PV_A(j) QK_A(j+1) PV_B(j) QK_B(j+1) | ...
//               so the tensor core works on one tile while the other tile's
//               softmax runs.  S = Q K^T lands in the tile's TMEM score
//               buffer; O += P V reads P from TMEM (the "TS" form) and V as an
//               MN-major 128-byte-swizzled shared-memory operand.  Operand
//               descriptors are built once and advanced by constants, and
//               the role runs on one lane with scalar waits, so the issuing
//               thread spends as few cycles as possible outside MMAs (the
//               tensor core's instruction queue is shallow).
//   warps 4-7   softmax of tile A, warps 8-11 of tile B: thread r owns TMEM
//               lane r = query row r; scores are loaded 128 at a time, masked
//               (causal, window, range) only on tiles that need it, the
//               running max is moved (and O rescaled in TMEM) only when it
//               grows by more than 2^8, and P is written back as bf16/fp16
//               pairs over the first 64 columns of the score buffer, 16
//               columns at a time; at the end O is normalised and stored.
//   warps 2-3   idle, except over an fp8 (E4M3) cache: there the producer
//               loads each tile's 8-bit codes (one plain box of D bytes x
//               block_size rows per cache block), and these two warps widen
//               them to fp16 in the 128-byte-swizzled layout the MMA reads
//               (E4M3 is a subset of fp16, so the codes are exact), then
//               release the stage to the MMA thread.  The MMAs then run on
//               fp16 operands: bf16 queries are rewritten in place as fp16
//               times a CTA-wide power of two 2^-e chosen from their largest
//               magnitude (exact scaling, no overflow), and k_scale * 2^e
//               joins the softmax scale; P is written as fp16 and v_scale
//               multiplies the output.  With D = 128 the codes land in the
//               stage's upper 64-column region and are widened in place, row
//               by row (a row is read completely before it is rewritten);
//               with D = 64 they have their own staging area.
// TMEM: S_A [0,128), S_B [128,256), O_A [256, 256+D), O_B [384, 384+D).
// Causal tile skipping: each query tile only visits the key tiles its rows
// can see; CTAs are ordered so the tiles with the most keys start first.
// Every wait is bounded; a timeout raises a CTA-wide abort flag, the roles
// stop, in-flight copies and MMAs are drained, TMEM is freed.
#include <cuda_fp8.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

struct PrefillArgs {
  void *out;
  const uint16_t *query;
  const int32_t *cu_q;
  const int32_t *cu_k;
  const int32_t *block_tables;
  const float *alibi;
  int64_t num_blocks;
  int64_t num_q_tokens;  // rows of query / out
  int num_seqs, max_blocks_per_seq;
  int H, KVH, QPK, BS, window, non_causal;
  float scale_log2;  // scale * log2(e) (* k_scale over an fp8 cache)
  float v_scale;     // 1, or the fp8 cache's value scale
};

namespace pf {

constexpr int BM = 128, BN = 128;
constexpr int NSTK = 2, NSTV = 2;  // K and V pipeline stages (a third K stage measured no faster)
constexpr int kThreads = 384;

template <int D, bool KV8 = false>
struct Lay {
  static constexpr int REG = 128 * 128;  // one 64-column region of 128 rows
  static constexpr int NREG = D / 64;
  static constexpr int TILE = REG * NREG;
  static constexpr int TILE8 = BN * D;  // one key tile of 8-bit codes
  // 16-bit K / V stages.  Over an fp8 cache the K codes are the QK operand
  // as they land (N8K staging areas, no 16-bit K stage); the V codes land in
  // N8V staging areas, each refilled as soon as its codes were widened into
  // one of the NV 16-bit V stages.
  static constexpr int NK = KV8 ? 0 : NSTK, NV = KV8 ? 2 : NSTV;
  static constexpr int N8K = 3, N8V = 2;
  static constexpr int OFF_Q = 0;  // two Q tiles
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NK * TILE;
  static constexpr int OFF_STG = OFF_V + NV * TILE;  // N8K K code tiles, then N8V V
  static constexpr int OFF_BAR = OFF_STG + (KV8 ? (N8K + N8V) * TILE8 : 0);
  // B_KF / B_VF: stage ready for the MMA; B_EK / B_EV: stage consumed by the
  // MMA; B_K8F / B_V8F: codes landed; B_E8K: K codes consumed by the MMA;
  // B_E8V: V codes widened; B_QS: a query tile's largest magnitude
  // gathered; B_Q2: its E4M3 terms ready
  static constexpr int B_Q = 0, B_KF = 1, B_VF = B_KF + NK, B_EK = B_VF + NV, B_EV = B_EK + NK,
                       B_SF = B_EV + NV, B_PF = B_SF + 2, B_O = B_PF + 2, B_FIN = B_O + 2,
                       B_Q2 = B_FIN + 1, B_QS = B_Q2 + 2, B_K8F = B_QS + 2, B_V8F = B_K8F + N8K,
                       B_E8K = B_V8F + N8V, B_E8V = B_E8K + N8K, NBAR = B_E8V + N8V;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  // + alignment slack; at least ~118 KB so that one CTA owns an SM (and all
  // of its tensor memory)
  static constexpr int ALLOC = (BYTES + 1024) > 118 * 1024 ? (BYTES + 1024) : 118 * 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                              volatile uint32_t *abort_flag, int64_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1u;
      record_error(PKV_ERR_TIMEOUT, where);
      return false;
    }
  }
}

// Warp-uniform verdict of a bounded wait performed by every lane.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity,
                                          volatile uint32_t *abort_flag, int64_t where) {
  const bool got = wait_or_abort(bar, parity, abort_flag, where);
  return __all_sync(0xffffffffu, got);
}

template <class T>
struct AB;
template <>
struct AB<BF16> {
  static constexpr int v = 1;
};
template <>
struct AB<FP16> {
  static constexpr int v = 0;
};


__device__ __forceinline__ uint32_t word4(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One query tile of the CTA: head, first row within the sequence, rows,
// and the half-open range of the CTA's key tiles it needs.
struct QTile {
  int head, q0, rows, j0, j1;
};

template <class T, int D, bool ALIBI, bool KV8>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
                  const __grid_constant__ CUtensorMap kvmap, int pair_heads) {
  using L = Lay<D, KV8>;
  using OPT = std::conditional_t<KV8, FP16, T>;  // MMA operand type (and P)
  constexpr int NK = L::NK, NV = L::NV;  // 16-bit K / V stages
  // barriers the K / V copies complete on, and how many stages they have
  constexpr int KFT = KV8 ? L::B_K8F : L::B_KF, VFT = KV8 ? L::B_V8F : L::B_VF;
  constexpr int NKT = KV8 ? L::N8K : NK, NVT = KV8 ? L::N8V : NV;
  // queries over an fp8 cache are rewritten as E4M3 terms by their softmax warps
  constexpr bool QCONV = KV8;
  constexpr int KEB = KV8 ? L::B_E8K : L::B_EK;  // K stage consumed by its QK products
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile uint32_t *abort_flag = misc + 1;

  // ---- which two tiles, and the key-tile range they span (CTA-uniform) ----
  const int b = blockIdx.y;
  const int zt = gridDim.z - 1 - blockIdx.z;  // heaviest tiles first
  QTile qt[2];
  if (pair_heads) {
    qt[0].head = 2 * blockIdx.x;
    qt[1].head = 2 * blockIdx.x + 1;
    qt[0].q0 = qt[1].q0 = zt * BM;
  } else {
    qt[0].head = qt[1].head = blockIdx.x;
    qt[0].q0 = zt * 2 * BM;
    qt[1].q0 = qt[0].q0 + BM;
  }
  const int qs = __ldg(a.cu_q + b), qe = __ldg(a.cu_q + b + 1);
  const int qb = qe - qs;
  const int Lb = __ldg(a.cu_k + b + 1) - __ldg(a.cu_k + b);
  if (qt[0].q0 >= qb) return;
  if (qs < 0 || qe > a.num_q_tokens || qb > Lb ||
      static_cast<int64_t>(Lb) > static_cast<int64_t>(a.max_blocks_per_seq) * a.BS) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(PKV_ERR_BOUNDS, b);
    return;
  }
  const int cb = Lb - qb;
  int kv_lo = 0x7fffffff, kv_end = 0;
  int lo_t[2], end_t[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    qt[x].rows = max(0, min(BM, qb - qt[x].q0));
    if (qt[x].rows > 0) {
      const int i_first = cb + qt[x].q0, i_last = i_first + qt[x].rows - 1;
      lo_t[x] = a.window > 0 ? max(0, i_first - a.window + 1) : 0;
      end_t[x] = a.non_causal ? Lb : i_last + 1;  // non-causal: every key
      kv_lo = min(kv_lo, lo_t[x]);
      kv_end = max(kv_end, end_t[x]);
    }
  }
  const int kv_start = kv_lo / BN * BN;
  const int ntiles = (kv_end - kv_start + BN - 1) / BN;
  // Key tiles are visited in step order 0 .. ntiles-1.  With ALiBi the step
  // order runs from the nearest key tile back to the farthest: the bias
  // slope * (j - i) falls tile by tile in that order, so a row's reference
  // max is set on its first (diagonal) tile and rarely has to move again,
  // where the far-to-near order moved it, and rescaled O, every tile of a
  // steep head.  phys(step) is the tile's index from kv_start.
  auto phys = [ntiles](int step) { return ALIBI ? ntiles - 1 - step : step; };
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    if (qt[x].rows > 0) {
      qt[x].j0 = (lo_t[x] / BN * BN - kv_start) / BN;
      qt[x].j1 = (end_t[x] - kv_start + BN - 1) / BN;
    } else {
      qt[x].j0 = qt[x].j1 = 0;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = qt[0].head / a.QPK;
  const int BS = a.BS;
  const int TB = BN / BS;
  const int64_t where = static_cast<int64_t>(b) * a.H + qt[0].head;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NBAR; ++i) {
      uint32_t count = (i == L::B_PF || i == L::B_PF + 1) ? 128 : 1;
      // the softmax warps of a tile release its E4M3 query terms; the V
      // stages and V staging areas are released by the two warps that widen
      // them (the K staging areas by an MMA commit)
      if (KV8 && (i == L::B_Q2 || i == L::B_Q2 + 1 || i == L::B_QS || i == L::B_QS + 1))
        count = 128;
      if (KV8 && ((i >= L::B_VF && i < L::B_VF + NV) || (i >= L::B_E8V && i < L::B_E8V + L::N8V)))
        count = 64;
      mbar_init(&bars[i], count);
    }
    misc[1] = 0;  // abort flag
    misc[2] = 0;  // K tiles issued
    misc[3] = 0;  // V tiles issued
    fence_mbar_init();
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kvmap);
  }
  if (warp == 1) tc5::tmem_alloc<512>(misc);
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int32_t *trow = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
    if (lane == 0) {
      const int nq = qt[1].rows > 0 ? 2 : 1;
      mbar_arrive_expect_tx(&bars[L::B_Q], nq * L::TILE);
      for (int x = 0; x < nq; ++x)
        for (int r = 0; r < L::NREG; ++r)
          tc5::tma_load_3d(smem + L::OFF_Q + x * L::TILE + r * L::REG, &qmap, &bars[L::B_Q],
                           64 * r, qt[x].head, qs + qt[x].q0);
    }
    // Lane l < TB handles cache block l of each key tile: its row coordinate
    // in the cache, or an out-of-range one (zero fill) outside the visible
    // range or for a bad table entry (recorded, never dereferenced).
    auto coord_of = [&](int j) -> int {
      int coord = -BS;
      if (lane < TB && j < ntiles) {
        const int lb = (kv_start + phys(j) * BN) / BS + lane;
        const int p0 = lb * BS;
        if (p0 < kv_end && p0 + BS > kv_lo) {
          const int pb = __ldg(trow + lb);
          if (pb < 0 || pb >= a.num_blocks)
            record_error(PKV_ERR_BOUNDS, static_cast<int64_t>(b) * a.max_blocks_per_seq + lb);
          else
            coord = pb * BS;
        }
      }
      return coord;
    };
    int next = coord_of(0);
    int jk = 0, jv = 0;  // K / V tiles issued
    for (int j = 0; j < ntiles; ++j) {
      const int coord = next;
      next = coord_of(j + 1);  // table entries of the next tile, fetched early
      if constexpr (KV8) {
        // codes into a staging area once the tile that used it was widened
        constexpr int N8K = L::N8K, N8V = L::N8V;
        const int sk8 = j % N8K, sv8 = j % N8V;
        if (j >= N8K &&
            !warp_wait(&bars[L::B_E8K + sk8], ((j / N8K) - 1) & 1, abort_flag, where))
          break;
        if (lane == 0) mbar_arrive_expect_tx(&bars[L::B_K8F + sk8], L::TILE8);
        __syncwarp();
        if (lane < TB)
          tma_load_4d(smem + L::OFF_STG + sk8 * L::TILE8 + lane * BS * D, &kvmap,
                      &bars[L::B_K8F + sk8], 0, g, coord, 0);
        jk = j + 1;
        if (j >= N8V &&
            !warp_wait(&bars[L::B_E8V + sv8], ((j / N8V) - 1) & 1, abort_flag, where))
          break;
        if (lane == 0) mbar_arrive_expect_tx(&bars[L::B_V8F + sv8], L::TILE8);
        __syncwarp();
        if (lane < TB)
          tma_load_4d(smem + L::OFF_STG + (N8K + sv8) * L::TILE8 + lane * BS * D, &kvmap,
                      &bars[L::B_V8F + sv8], 0, g, coord, 1);
        jv = j + 1;
      } else {
        const int sk = j % NK;
        if (j >= NK && !warp_wait(&bars[L::B_EK + sk], ((j / NK) - 1) & 1, abort_flag, where))
          break;
        if (lane == 0) mbar_arrive_expect_tx(&bars[L::B_KF + sk], L::TILE);
        __syncwarp();
        if (lane < TB) {
          uint8_t *kd = smem + L::OFF_K + sk * L::TILE + lane * BS * 128;
          for (int r = 0; r < L::NREG; ++r)
            tma_load_4d(kd + r * L::REG, &kvmap, &bars[L::B_KF + sk], 64 * r, g, coord, 0);
        }
        jk = j + 1;
        const int sv = j % NV;
        if (j >= NV && !warp_wait(&bars[L::B_EV + sv], ((j / NV) - 1) & 1, abort_flag, where))
          break;
        if (lane == 0) mbar_arrive_expect_tx(&bars[L::B_VF + sv], L::TILE);
        __syncwarp();
        if (lane < TB) {
          uint8_t *vd = smem + L::OFF_V + sv * L::TILE + lane * BS * 128;
          for (int r = 0; r < L::NREG; ++r)
            tma_load_4d(vd + r * L::REG, &kvmap, &bars[L::B_VF + sv], 64 * r, g, coord, 1);
        }
        jv = j + 1;
      }
    }
    if (lane == 0) {
      misc[2] = static_cast<uint32_t>(jk);
      misc[3] = static_cast<uint32_t>(jv);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // One thread: the tensor core's instruction queue is shallow, so every
    // cycle this thread spends outside an MMA is a cycle the tensor core may
    // idle.  Waits are scalar; there is no warp-wide synchronisation here.
    // QK over an fp8 cache: kind::f8f6f4, E4M3 query terms x E4M3 key codes
    constexpr uint32_t ID_QK = tc5::idesc_f16(KV8 ? 0 : AB<OPT>::v, 0, BM, BN);
    constexpr uint32_t ID_PV = tc5::idesc_f16(AB<OPT>::v, 1, BM, D);
    // Operand descriptors are built once; an MMA only adds a compile-time
    // offset (in 16-byte units) to a base.  8-bit operands are K-major rows
    // of D bytes: 128-byte swizzle for D = 128, 64-byte for D = 64.
    auto sdesc8 = [&](uint32_t off) -> uint64_t {
      return D == 128 ? tc5::sdesc_sw128(sbase + off, 16, 1024) : tc5::sdesc_sw64(sbase + off, 16, 512);
    };
    const uint64_t q_desc = KV8 ? sdesc8(L::OFF_Q) : tc5::sdesc_sw128(sbase + L::OFF_Q, 16, 1024);
    const uint64_t k_desc = KV8 ? sdesc8(L::OFF_STG) : tc5::sdesc_sw128(sbase + L::OFF_K, 16, 1024);
    const uint64_t v_desc = tc5::sdesc_sw128(sbase + L::OFF_V, L::REG, 1024);
    const int j0A = qt[0].j0, j1A = qt[0].j1, j0B = qt[1].j0, j1B = qt[1].j1;
    auto active = [&](int x, int j) {
      const int p = phys(j);
      return x == 0 ? (p >= j0A && p < j1A) : (p >= j0B && p < j1B);
    };
    int k_ready = -1;  // highest key tile known to have landed
    auto need_k = [&](int j) -> bool {
      if (j <= k_ready) return true;
      if (!wait_or_abort(&bars[KFT + j % NKT], (j / NKT) & 1, abort_flag, where))
        return false;
      tc5::fence_after_sync();
      k_ready = j;
      return true;
    };
    auto qk = [&](int x, int j) {
      const uint64_t qb = q_desc + static_cast<uint64_t>((x * L::TILE) >> 4);
      const uint32_t sb = tmem + x * 128;
      if constexpr (KV8) {
        // S = Q_hi K^T + Q_lo K^T, 32 codes (32 bytes) per k-step
        const uint64_t kb = k_desc + static_cast<uint64_t>(((j % L::N8K) * L::TILE8) >> 4);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int k = 0; k < D / 32; ++k)
            tc5::mma_ss_f8(sb, qb + static_cast<uint64_t>((t * BM * D + k * 32) >> 4),
                           kb + static_cast<uint64_t>(k * 2), ID_QK, (t | k) ? 1u : 0u);
      } else {
        const uint64_t kb = k_desc + static_cast<uint64_t>(((j % NK) * L::TILE) >> 4);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t off = static_cast<uint64_t>(((k / 4) * L::REG + (k % 4) * 32) >> 4);
          tc5::mma_ss(sb, qb + off, kb + off, ID_QK, k > 0 ? 1u : 0u);
        }
      }
      tc5::commit(&bars[L::B_SF + x]);
    };
    bool ok = wait_or_abort(&bars[QCONV ? L::B_Q2 : L::B_Q], 0, abort_flag, where);
    if (QCONV && ok && qt[1].rows > 0) ok = wait_or_abort(&bars[L::B_Q2 + 1], 0, abort_flag, where);
    if (ok && ntiles > 0) {
      ok = need_k(0);
      if (ok) {
        if (active(0, 0)) qk(0, 0);
        if (active(1, 0)) qk(1, 0);
        tc5::commit(&bars[KEB + 0]);  // K(0) free once its QKs finish
      }
    }
    int pf_a = 0, pf_b = 0;  // P tiles consumed per query tile
    // PV of tile x for key tile j, then the look-ahead QK of tile x
    auto step = [&](int x, int j, int sv, int &pf) -> bool {
      if (active(x, j)) {
        if (!wait_or_abort(&bars[L::B_PF + x], pf & 1, abort_flag, where)) return false;
        tc5::fence_after_sync();
        const uint32_t pb = tmem + x * 128;
        const uint32_t ob = tmem + 256 + x * 128;
        const uint64_t vb = v_desc + static_cast<uint64_t>((sv * L::TILE) >> 4);
        const uint32_t acc0 = pf > 0 ? 1u : 0u;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)  // 16 keys = 2048 bytes of V per step
          tc5::mma_ts(ob, pb + k * 8, vb + static_cast<uint64_t>(k * 128), ID_PV,
                      k > 0 ? 1u : acc0);
        tc5::commit(&bars[L::B_O + x]);
        ++pf;
      }
      if (j + 1 < ntiles && active(x, j + 1)) {
        if (!need_k(j + 1)) return false;
        qk(x, j + 1);
      }
      return true;
    };
    for (int j = 0; ok && j < ntiles; ++j) {
      const int sv = j % NV;
      if (!wait_or_abort(&bars[L::B_VF + sv], (j / NV) & 1, abort_flag, where)) break;
      // Positions past the sequence end inside its last cache block hold
      // whatever the cache holds there (possibly non-finite); their P is
      // exactly 0, but 0 * NaN is NaN, so those V rows are zeroed before the
      // PV product reads them.  Whole blocks past the end came in as zeros.
      const int kv0 = kv_start + phys(j) * BN;
      const int zr = Lb - kv0;
      if (zr > 0 && zr < BN && zr % BS != 0) {
        const int ze = min(BN, (zr / BS + 1) * BS);
        uint8_t *vt = smem + L::OFF_V + sv * L::TILE;
        for (int r = 0; r < L::NREG; ++r)
          for (int c = zr * 8; c < ze * 8; ++c)
            *reinterpret_cast<uint4 *>(vt + r * L::REG + c * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      if (!step(0, j, sv, pf_a) || !step(1, j, sv, pf_b)) break;
      tc5::commit(&bars[L::B_EV + sv]);                                  // V(j) after its PVs
      if (j + 1 < ntiles) tc5::commit(&bars[KEB + (j + 1) % NKT]);  // K(j+1) after its QKs
    }
    // every MMA this thread issued has completed before TMEM is released
    tc5::commit(&bars[L::B_FIN]);
    mbar_wait_bounded(&bars[L::B_FIN], 0, where);
  } else if (KV8 && (warp == 2 || warp == 3)) {
    // ------------------------------------------------------------ fp8 widening
    const int cw = warp - 2;
    bool ok = true;
    // Per key tile the V codes are widened by warps 2 and 3, each taking
    // half the rows (the K codes are the QK operand as they are).
    // Lane (row r0, column group cc) widens 16 codes (one 16-byte load of
    // the swizzled code rows) into two 16-byte chunks of the swizzled fp16
    // tile; lanes of the upper column half store their two chunks in the
    // opposite order, so that the 8 lanes of one row never hit the same bank
    // group in one store.
    constexpr int LPR = D / 16, RPI = 32 / LPR;  // lanes per row, rows per pass
    constexpr int ROWS = BM / 2;  // rows each converter warp widens
    const int cc = lane % LPR, r0 = lane / LPR;
    const int row_base = cw * ROWS;
    const int swap = (cc >= LPR / 2) ? 1 : 0;
    // this lane's row r = row_base + RPI * it + r0 has swizzle phase
    // r & 7 = r0 ^ ((RPI * it) & 7) for 128-byte rows (D = 128) and
    // (r >> 1) & 3 = (r0 >> 1) & 3 for 64-byte rows (D = 64)
    auto code_chunk = [&](int ph) {
      return D == 128 ? (cc ^ r0 ^ (4 * ph)) : (cc ^ ((r0 >> 1) & 3));
    };
    auto widen = [&](int j) -> bool {
      const int s = j % NV, s8 = j % L::N8V;
      if (!warp_wait(&bars[L::B_V8F + s8], (j / L::N8V) & 1, abort_flag, where)) return false;
      // the fp16 stage is free once the MMAs of the tile that used it are done
      if (j >= NV && !warp_wait(&bars[L::B_EV + s], ((j / NV) - 1) & 1, abort_flag, where))
        return false;
      const uint8_t *src = smem + L::OFF_STG + (L::N8K + s8) * L::TILE8;
      uint8_t *dst = smem + L::OFF_V + s * L::TILE;
      // the lane's chunk addresses are a lane-constant base plus a
      // compile-time offset per pass
      const uint8_t *ls[2];
      uint8_t *ld = dst + (cc / 4) * L::REG + (row_base + r0) * 128;
      const int k0 = (2 * cc) % 8;
      uint8_t *pa[2], *pb[2];  // [phase 0 / 4]: first, second chunk
#pragma unroll
      for (int ph = 0; ph < 2; ++ph) {
        ls[ph] = src + (row_base + r0) * D + code_chunk(ph) * 16;
        pa[ph] = ld + ((k0 ^ r0 ^ (4 * ph)) * 16);
        pb[ph] = ld + (((k0 + 1) ^ r0 ^ (4 * ph)) * 16);
        if (swap) {  // store order flipped for the upper column half
          uint8_t *t = pa[ph];
          pa[ph] = pb[ph];
          pb[ph] = t;
        }
      }
#pragma unroll
      for (int it = 0; it < ROWS / RPI; ++it) {
        const int ph = ((RPI * it) & 7) ? 1 : 0;
        const uint4 u = *reinterpret_cast<const uint4 *>(ls[ph] + it * RPI * D);
        const uint2 h0 = e4m3x4_to_h4(u.x), h1 = e4m3x4_to_h4(u.y);
        const uint2 h2 = e4m3x4_to_h4(u.z), h3 = e4m3x4_to_h4(u.w);
        // dims 16cc .. 16cc+7 and 16cc+8 .. 16cc+15 (swapped with the order)
        const uint4 c0 = make_uint4(h0.x, h0.y, h1.x, h1.y);
        const uint4 c1 = make_uint4(h2.x, h2.y, h3.x, h3.y);
        *reinterpret_cast<uint4 *>(pa[ph] + it * RPI * 128) = swap ? c1 : c0;
        *reinterpret_cast<uint4 *>(pb[ph] + it * RPI * 128) = swap ? c0 : c1;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[L::B_VF + s]);
      mbar_arrive(&bars[L::B_E8V + s8]);  // staging area free again
      return true;
    };
    for (int j = 0; ok && j < ntiles; ++j) ok = widen(j);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int x = warp >= 8 ? 1 : 0;
    const QTile t = x ? qt[1] : qt[0];
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t sb = tmem + lane_base + x * 128;
    const uint32_t ob = tmem + lane_base + 256 + x * 128;
    const int pos = cb + t.q0 + row;
    const int lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
    const int hi = a.non_causal ? Lb - 1 : pos;  // last visible key
    float sl2 = a.scale_log2;
    const float slope = ALIBI ? __ldg(a.alibi + t.head) * kLog2e : 0.f;
    // running max m: in the log2 domain with ALiBi; in raw-score units
    // without (then scores are scaled inside the exponent's FMA)
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    if constexpr (QCONV) {
      // This tile's queries become two E4M3 terms hi + lo of q * 2^-e, e
      // chosen from their largest magnitude (largest |q| * 2^-e in
      // [2^7, 2^8): both terms inside E4M3's range; exact power-of-two
      // scaling), written over the tile as two K-major tiles of D-byte rows
      // (hi, then lo) in the swizzled layout of the key codes; 2^e joins the
      // score scale.  The four warps exchange their maxima through an
      // mbarrier, which also tells every warp that the whole tile has been
      // read before any of it is overwritten (bounded waits: no barrier can
      // strand a warp).
      constexpr int CH = L::TILE / 16 / 128;  // 16-byte chunks per thread
      int e = 0;
      ok = warp_wait(&bars[L::B_Q], 0, abort_flag, where);
      uint8_t *qt8 = smem + L::OFF_Q + x * L::TILE;
      const uint4 *q4 = reinterpret_cast<const uint4 *>(qt8);
      const int tid = (warp & 3) * 32 + lane;
      uint4 qv[CH];
      uint32_t am = 0;  // largest |q| (fp32 bit pattern)
      if (ok) {
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          qv[i] = q4[tid + 128 * i];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = T::to_f2(word4(qv[i], k));
            am = max(am, max(__float_as_uint(fabsf(f.x)), __float_as_uint(fabsf(f.y))));
          }
        }
        am = __reduce_max_sync(0xffffffffu, am);
        if (lane == 0) misc[8 + x * 4 + (warp & 3)] = am;
        mbar_arrive(&bars[L::B_QS + x]);
        ok = warp_wait(&bars[L::B_QS + x], 0, abort_flag, where);
      }
      if (ok) {
        am = max(max(misc[8 + x * 4], misc[9 + x * 4]), max(misc[10 + x * 4], misc[11 + x * 4]));
        const int E = static_cast<int>(am >> 23);
        e = E == 0 ? 0 : min(64, max(-64, E - 134));
        const float mul = __int_as_float((127 - e) << 23);
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          // chunk c of the 16-bit tile: 64-dim region, row, logical chunk
          const int c = tid + 128 * i;
          const int r = c / (L::REG / 16), R = (c % (L::REG / 16)) / 8;
          const int d0 = 64 * r + 8 * ((c % 8) ^ (R & 7));  // its first of 8 dims
          float v[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = T::to_f2(word4(qv[i], k));
            v[2 * k] = f.x * mul;
            v[2 * k + 1] = f.y * mul;
          }
          uint32_t h0, l0, h1, l1;
          split_e4m3x4(v[0], v[1], v[2], v[3], h0, l0);
          split_e4m3x4(v[4], v[5], v[6], v[7], h1, l1);
          // its 8 codes at byte d0 of row R of the D-byte swizzled rows
          const int off = D == 128 ? R * 128 + ((((d0 >> 4) ^ (R & 7)) << 4) | (d0 & 8))
                                   : R * 64 + ((((d0 >> 4) ^ ((R >> 1) & 3)) << 4) | (d0 & 8));
          *reinterpret_cast<uint2 *>(qt8 + off) = make_uint2(h0, h1);
          *reinterpret_cast<uint2 *>(qt8 + BM * D + off) = make_uint2(l0, l1);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[L::B_Q2 + x]);
      }
      sl2 *= __int_as_float((127 + e) << 23);
    }
    const int n = t.j1 - t.j0;
    for (int k = 0; ok && k < n; ++k) {
      const int j = ALIBI ? t.j1 - 1 - k : t.j0 + k;  // this tile's k-th key tile
      if (!warp_wait(&bars[L::B_SF + x], k & 1, abort_flag, where)) {
        ok = false;
        break;
      }
      tc5::fence_after_sync();
      uint32_t raw[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tc5::tmem_ld32(sb + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(raw + 32 * c));
      tc5::tmem_ld_wait();
      const int kv0 = kv_start + j * BN;
      const bool full = (kv0 + BN - 1 <= hi) && (kv0 >= lo);
      if (__any_sync(0xffffffffu, !full)) {  // every lane enters: the votes below span the warp
        // per 32-key chunk the warp's rows agree that it is wholly visible
        // (nothing to do), wholly hidden (all -inf) or needs the per-key mask
        // (a row whose whole tile is visible finds every chunk visible)
        const int vlo = lo - kv0, vhi = hi - kv0;  // visible offsets [vlo, vhi]
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          const bool some_hidden = !__all_sync(0xffffffffu, 32 * c >= vlo && 32 * c + 31 <= vhi);
          const bool all_hidden = __all_sync(0xffffffffu, 32 * c > vhi || 32 * c + 31 < vlo);
          const int mlo = all_hidden ? BN : vlo, mhi = all_hidden ? -1 : vhi;
          if (some_hidden) {
#pragma unroll
            for (int e = 32 * c; e < 32 * c + 32; ++e)
              if (e > mhi || e < mlo) raw[e] = __float_as_uint(-INFINITY);
          }
        }
      }
      const float unit = ALIBI ? 1.f : sl2;  // log2 units per unit of m
      // p = 2^(x - mu) over the tile, written to TMEM as P; returns the row
      // sum.  With ALiBi x is already scaled (and biased); without, the scale
      // is folded into the pair FMA.
      auto exps = [&](float mu) -> float {
        const unsigned long long mul2 = ALIBI ? f2pack(1.f, 1.f) : f2pack(sl2, sl2);
        const unsigned long long negmu2 = f2pack(-mu, -mu);
        unsigned long long ps2[4] = {0ull, 0ull, 0ull, 0ull};  // packed partial sums
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0, x1;
            f2unpack(ffma2(f2pack(__uint_as_float(raw[32 * c + e]),
                                  __uint_as_float(raw[32 * c + e + 1])),
                           mul2, negmu2),
                     x0, x1);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            ps2[(e / 2) & 3] = fadd2(ps2[(e / 2) & 3], f2pack(p0, p1));
            pk[e / 2] = OPT::from_f2(p0, p1);
          }
          tc5::tmem_st16(sb + 16 * c, pk);
        }
        float ps0, ps1;
        f2unpack(fadd2(fadd2(ps2[0], ps2[1]), fadd2(ps2[2], ps2[3])), ps0, ps1);
        return ps0 + ps1;
      };
      // ALiBi: p = 2^(s * sl2 + (slope * e + A)) for the tile's key offsets
      // e = j - kv0, A = slope * (kv0 - i) - mu: the bias is folded into the
      // exponent's FMA (its terms from immediate offsets), raw untouched.
      auto exps_alibi = [&](float A) -> float {
        const unsigned long long mul2 = f2pack(sl2, sl2);
        unsigned long long ps2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = 32 * c + e;
            const float b0 = fmaf(slope, static_cast<float>(col), A);
            const float b1 = fmaf(slope, static_cast<float>(col + 1), A);
            float x0, x1;
            f2unpack(ffma2(f2pack(__uint_as_float(raw[col]), __uint_as_float(raw[col + 1])),
                           mul2, f2pack(b0, b1)),
                     x0, x1);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            ps2[(e / 2) & 1] = fadd2(ps2[(e / 2) & 1], f2pack(p0, p1));
            pk[e / 2] = OPT::from_f2(p0, p1);
          }
          tc5::tmem_st16(sb + 16 * c, pk);
        }
        float ps0, ps1;
        f2unpack(fadd2(ps2[0], ps2[1]), ps0, ps1);
        return ps0 + ps1;
      };
      // The reference m moves lazily, so the tile's max only decides
      // whether it must move: the exponents are first taken against m as it
      // stands, and only a row whose sum is out of range (m not set yet, or a
      // p too large for an fp16 P) sends its warp through the max and a
      // second pass.  With ALiBi the nearest key tile comes first, so m is
      // set where the bias peaks and the later (farther) tiles rarely pass it.
      float alpha = 1.f;
      bool resc = false;
      float ps = 0.f;
      bool slow = m == -INFINITY;
      if (!__any_sync(0xffffffffu, slow)) {
        ps = ALIBI ? exps_alibi(slope * static_cast<float>(kv0 - pos) - m) : exps(m * unit);
        slow = !(ps <= 32768.f);
      }
      if (__any_sync(0xffffffffu, slow)) {
        if constexpr (ALIBI) {
          // x = s * scale * log2e + slope * log2e * (j - i), in pairs
          const float b0 = slope * static_cast<float>(kv0 - pos);
          const unsigned long long sl2x2 = f2pack(sl2, sl2);
#pragma unroll
          for (int e = 0; e < BN; e += 2) {
            const unsigned long long bias = f2pack(fmaf(slope, static_cast<float>(e), b0),
                                                   fmaf(slope, static_cast<float>(e + 1), b0));
            float v0, v1;
            f2unpack(ffma2(f2pack(__uint_as_float(raw[e]), __uint_as_float(raw[e + 1])), sl2x2,
                           bias),
                     v0, v1);
            raw[e] = __float_as_uint(v0);
            raw[e + 1] = __float_as_uint(v1);
          }
        }
        // 8 independent 3-input max chains, then a small tree
        float pm[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) pm[q] = -INFINITY;
#pragma unroll
        for (int e = 0; e < BN; e += 2)
          pm[(e / 2) & 7] =
              fmax3(pm[(e / 2) & 7], __uint_as_float(raw[e]), __uint_as_float(raw[e + 1]));
        const float mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]),
                               fmaxf(pm[6], pm[7]));
        // move the max when it grows by more than 8 (2^8 in p)
        if (m == -INFINITY) {
          m = mx;
        } else if ((mx - m) * unit > 8.f) {
          alpha = fast_exp2((m - mx) * unit);
          m = mx;
          resc = true;
        }
        tc5::tmem_st_wait();  // a first pass's P is written before it is replaced
        ps = exps(m == -INFINITY ? 0.f : m * unit);
      }
      l = l * alpha + ps;
      if (__any_sync(0xffffffffu, resc)) {
        // O_x holds PV of the previous key tile once it has completed
        if (!warp_wait(&bars[L::B_O + x], (k - 1) & 1, abort_flag, where)) {
          ok = false;
          break;
        }
        tc5::fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc5::tmem_ld32(ob + 32 * c, o);
          tc5::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc5::tmem_st32(ob + 32 * c, o);
        }
      }
      tc5::tmem_st_wait();
      tc5::fence_before_sync();
      mbar_arrive(&bars[L::B_PF + x]);
    }
    if (ok && n > 0 && warp_wait(&bars[L::B_O + x], (n - 1) & 1, abort_flag, where)) {
      tc5::fence_after_sync();
      const float inv = l > 0.f ? (KV8 ? a.v_scale : 1.f) / l : 0.f;
      const bool valid = row < t.rows;
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) +
                                             (static_cast<int64_t>(qs + t.q0 + row) * a.H + t.head) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc5::tmem_ld32(ob + 32 * c, o);
        tc5::tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = T::from_f2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[c * 4 + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
    }
    tc5::fence_before_sync();
  }

  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // let every copy that was issued land before the CTA's memory goes away
    mbar_wait_bounded(&bars[L::B_Q], 0, where);
    const int nk = static_cast<int>(misc[2]), nv = static_cast<int>(misc[3]);
    for (int s = 0; s < NKT; ++s) {
      const int t = nk - 1 - ((nk - 1 - s) % NKT + NKT) % NKT;  // last K tile of stage s
      if (t >= 0 && t % NKT == s) mbar_wait_bounded(&bars[KFT + s], (t / NKT) & 1, where);
    }
    for (int s = 0; s < NVT; ++s) {
      const int t = nv - 1 - ((nv - 1 - s) % NVT + NVT) % NVT;
      if (t >= 0 && t % NVT == s) mbar_wait_bounded(&bars[VFT + s], (t / NVT) & 1, where);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc5::fence_after_sync();
    tc5::tmem_dealloc<512>(tmem);
  }
}

template <class T, int D, bool ALIBI, bool KV8>
cudaError_t launch(const PrefillArgs &a, int max_query_len, const CUtensorMap &qmap,
                   const CUtensorMap &kvmap, cudaStream_t stream) {
  const size_t smem = Lay<D, KV8>::ALLOC;
  auto kern = prefill_tc_kernel<T, D, ALIBI, KV8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int pair = (a.QPK % 2 == 0) ? 1 : 0;
  const int tiles = (max_query_len + BM - 1) / BM;
  dim3 grid(pair ? a.H / 2 : a.H, a.num_seqs, pair ? tiles : (tiles + 1) / 2);
  kern<<<grid, kThreads, smem, stream>>>(a, qmap, kvmap, pair);
  return cudaGetLastError();
}

template <class T, int D>
cudaError_t launch_any(const PrefillArgs &a, int max_query_len, const CUtensorMap &qmap,
                       const CUtensorMap &kvmap, bool kv8, cudaStream_t stream) {
  if (kv8)
    return a.alibi ? launch<T, D, true, true>(a, max_query_len, qmap, kvmap, stream)
                   : launch<T, D, false, true>(a, max_query_len, qmap, kvmap, stream);
  return a.alibi ? launch<T, D, true, false>(a, max_query_len, qmap, kvmap, stream)
                 : launch<T, D, false, false>(a, max_query_len, qmap, kvmap, stream);
}

}  // namespace pf

cudaError_t launch_prefill(void *out, const void *query, int64_t num_q_tokens, int num_seqs,
                           const int32_t *cu_q, const int32_t *cu_k, int max_query_len,
                           int max_seq_len, const void *kv_cache, const int32_t *block_tables,
                           int max_blocks_per_seq, const Geometry &g, cudaStream_t stream) {
  (void)max_seq_len;
  PrefillArgs a{};
  a.out = out;
  a.query = static_cast<const uint16_t *>(query);
  a.cu_q = cu_q;
  a.cu_k = cu_k;
  a.block_tables = block_tables;
  a.alibi = g.alibi;
  a.num_blocks = g.num_blocks;
  a.num_q_tokens = num_q_tokens;
  a.num_seqs = num_seqs;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.H = g.H;
  a.KVH = g.KVH;
  a.QPK = g.QPK;
  a.BS = g.BS;
  a.window = g.window;
  a.non_causal = g.non_causal;
  a.scale_log2 = g.scale * kLog2e * g.k_scale;
  a.v_scale = g.v_scale;
  const bool bf = g.dtype == PKV_BF16;
  // Q: (D, H, tokens); cache: (D, KVH, NB * BS tokens, 2 halves); 64-element
  // (128-byte) inner boxes with the 128-byte swizzle the MMA descriptors use.
  const CUtensorMapDataType dt =
      bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap qmap, kvmap;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.D), static_cast<cuuint64_t>(g.H),
                                static_cast<cuuint64_t>(num_q_tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.D) * 2,
                                   static_cast<cuuint64_t>(g.H) * g.D * 2};
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(pf::BM)};
    if (encode_tensor_map(&qmap, dt, 3, const_cast<void *>(query), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // 16-bit cache: 64-element swizzled boxes; fp8 cache: one box of the
    // whole D-byte row per cache block, swizzled by its row length (the key
    // codes are the QK operand as they land; the widening warps read the
    // value codes through the same swizzle)
    const cuuint64_t eb = static_cast<cuuint64_t>(g.elem_bytes);
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.D), static_cast<cuuint64_t>(g.KVH),
                                static_cast<cuuint64_t>(g.num_blocks * g.BS), 2};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.D) * eb,
                                   static_cast<cuuint64_t>(g.row_elems) * eb,
                                   static_cast<cuuint64_t>(g.num_blocks * g.block_elems) * eb};
    const cuuint32_t box[4] = {g.fp8 ? static_cast<cuuint32_t>(g.D) : 64u, 1,
                               static_cast<cuuint32_t>(g.BS), 1};
    const CUtensorMapSwizzle swz = !g.fp8 || g.D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                         : CU_TENSOR_MAP_SWIZZLE_64B;
    if (encode_tensor_map(&kvmap, g.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : dt, 4,
                          const_cast<void *>(kv_cache), dims, strides, box, swz) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (g.D == 128)
    return bf ? pf::launch_any<BF16, 128>(a, max_query_len, qmap, kvmap, g.fp8, stream)
              : pf::launch_any<FP16, 128>(a, max_query_len, qmap, kvmap, g.fp8, stream);
  if (g.D == 64)
    return bf ? pf::launch_any<BF16, 64>(a, max_query_len, qmap, kvmap, g.fp8, stream)
              : pf::launch_any<FP16, 64>(a, max_query_len, qmap, kvmap, g.fp8, stream);
  return cudaErrorInvalidValue;
}

cudaError_t read_device_error_prefill(unsigned long long *out) {
  return read_and_clear_unit_error(out);
}

}  // namespace pkv
