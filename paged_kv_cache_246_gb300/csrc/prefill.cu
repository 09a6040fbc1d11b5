// Varlen causal prefill over the paged cache, with or without a cached
// context (chunked prefill).
//
// What is computed (xformers.py XFormersImpl.forward -> forward_prefix and
// _run_memory_efficient_xformers_forward; cpu_attn flash_attn_varlen_func):
// sequence b has L_b = cu_k[b+1] - cu_k[b] tokens of which the last
// q_b = cu_q[b+1] - cu_q[b] are query rows; row t sits at position
// i = (L_b - q_b) + t and attends to keys lo(i) <= j <= i of its sequence,
// all read through the block table:
//     s_j = scale * q.k_j + slope_h * (j - i),   out = softmax(s) . V.
//
// This unit holds the warp-level tensor-core kernel: CTA = (query head,
// sequence, 64-row query tile), 4 warps x 16 rows, 64-key tiles gathered
// through the block table with cp.async into XOR-swizzled shared memory
// (double-buffered), m16n8k16 MMAs for q.k and p.V with fp32 accumulators,
// online softmax in registers in the log2 domain.  Tiles are visited from
// the last query tile of every (head, sequence) to the first, so the longest
// tiles start first.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

struct PrefillArgs {
  void *out;
  const uint16_t *query;
  const uint16_t *k_half;
  const uint16_t *v_half;
  const int32_t *cu_q;
  const int32_t *cu_k;
  const int32_t *block_tables;
  const float *alibi;
  int64_t num_blocks;
  int64_t num_q_tokens;  // rows of query / out
  int num_seqs, max_blocks_per_seq;
  int H, KVH, QPK, BS, window;
  float scale_log2;
};

// Per-(sequence, query tile) facts shared by both kernels; false if the tile
// is empty or the sequence's metadata is inconsistent (recorded).
struct TileSpan {
  int qs, qb, Lb, cb, q0, q_rows, kv_start, kv_end, kv_lo, ntiles;
};

template <int BM_, int BN_>
__device__ __forceinline__ bool tile_span(const PrefillArgs &a, int b, int tile, bool report,
                                          TileSpan &t) {
  t.q0 = tile * BM_;
  t.qs = __ldg(a.cu_q + b);
  const int qe = __ldg(a.cu_q + b + 1);
  t.qb = qe - t.qs;
  t.Lb = __ldg(a.cu_k + b + 1) - __ldg(a.cu_k + b);
  if (t.q0 >= t.qb) return false;
  if (t.qs < 0 || qe > a.num_q_tokens || t.qb > t.Lb ||
      static_cast<int64_t>(t.Lb) > static_cast<int64_t>(a.max_blocks_per_seq) * a.BS) {
    if (report) record_error(PKV_ERR_BOUNDS, b);
    return false;
  }
  t.cb = t.Lb - t.qb;
  t.q_rows = min(BM_, t.qb - t.q0);
  const int i_first = t.cb + t.q0, i_last = t.cb + t.q0 + t.q_rows - 1;
  t.kv_lo = a.window > 0 ? max(0, i_first - a.window + 1) : 0;
  t.kv_start = t.kv_lo / BN_ * BN_;
  t.kv_end = i_last + 1;
  t.ntiles = (t.kv_end - t.kv_start + BN_ - 1) / BN_;
  return true;
}

namespace mma_path {

constexpr int BM = 64;  // query rows per CTA
constexpr int BN = 64;  // keys per tile
constexpr int kThreads = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: zero-fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <class T>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<BF16>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<FP16>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk c of row r in a swizzled [rows][D] tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((r * (D / 8) + (c ^ (r & 7))) * 16);
}

template <class T, int D>
__global__ void __launch_bounds__(kThreads)
prefill_mma_kernel(const PrefillArgs a) {
  constexpr int ROWC = D / 8;
  constexpr int TILE_BYTES = BN * D * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + BM * D * 2;          // 2 buffers
  const uint32_t sV = sK + 2 * TILE_BYTES;      // 2 buffers

  const int h = blockIdx.x, b = blockIdx.y;
  const int tile = gridDim.z - 1 - blockIdx.z;
  TileSpan sp;
  if (!tile_span<BM, BN>(a, b, tile, threadIdx.x == 0 && h == 0, sp)) return;
  const int q0 = sp.q0, qs = sp.qs, cb = sp.cb, q_rows = sp.q_rows;
  const int kv_start = sp.kv_start, kv_end = sp.kv_end, ntiles = sp.ntiles;
  const int g = h / a.QPK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t *trow = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;

  // ---- async loads --------------------------------------------------------
  auto load_q = [&]() {
    for (int idx = tid; idx < BM * ROWC; idx += kThreads) {
      const int r = idx / ROWC, c = idx % ROWC;
      const bool v = r < q_rows;
      const uint16_t *src =
          a.query + (static_cast<int64_t>(qs + q0 + (v ? r : 0)) * a.H + h) * D + c * 8;
      cp_async16(sQ + swz<D>(r, c), src, v);
    }
  };
  auto load_kv = [&](int t, int buf) {
    const int kv0 = kv_start + t * BN;
    for (int idx = tid; idx < BN * ROWC; idx += kThreads) {
      const int r = idx / ROWC, c = idx % ROWC;
      const int j = kv0 + r;
      bool v = j < kv_end;
      int64_t slot = 0;
      if (v) {
        const int pb = __ldg(trow + j / a.BS);
        if (pb < 0 || pb >= a.num_blocks) {
          record_error(PKV_ERR_BOUNDS, static_cast<int64_t>(b) * a.max_blocks_per_seq + j / a.BS);
          v = false;
        } else {
          slot = static_cast<int64_t>(pb) * a.BS + j % a.BS;
        }
      }
      const int64_t off = (slot * a.KVH + g) * D + c * 8;
      cp_async16(sK + buf * TILE_BYTES + swz<D>(r, c), a.k_half + off, v);
      cp_async16(sV + buf * TILE_BYTES + swz<D>(r, c), a.v_half + off, v);
    }
  };

  load_q();
  load_kv(0, 0);
  cp_commit();

  // ---- per-thread state ---------------------------------------------------
  const int gr = lane >> 2, gc = lane & 3;
  const int r0 = warp * 16 + gr;  // tile rows owned: r0, r0 + 8
  const int pos0 = cb + q0 + r0, pos1 = pos0 + 8;
  const float slope = a.alibi ? __ldg(a.alibi + h) * kLog2e : 0.f;
  uint32_t qf[D / 16][4];
  float oacc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[n][e] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int lo0 = a.window > 0 ? max(0, pos0 - a.window + 1) : 0;
  const int lo1 = a.window > 0 ? max(0, pos1 - a.window + 1) : 0;

  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < ntiles) {
      load_kv(t + 1, buf ^ 1);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    if (t == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int r = warp * 16 + (lane & 15);
        const int c = ks * 2 + (lane >> 4);
        ldsm_x4(sQ + swz<D>(r, c), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    const uint32_t kb = sK + buf * TILE_BYTES, vb = sV + buf * TILE_BYTES;
    // ---- S = Q K^T (16 x 64 per warp) -------------------------------------
    float s[BN / 8][4];
#pragma unroll
    for (int n = 0; n < BN / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int np = 0; np < BN / 16; ++np) {
        const int key = np * 16 + (lane >> 4) * 8 + (lane & 7);
        const int c = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz<D>(key, c), b0, b1, b2, b3);
        mma16816<T>(s[2 * np], qf[ks], b0, b1);
        mma16816<T>(s[2 * np + 1], qf[ks], b2, b3);
      }
    }
    // ---- mask, ALiBi, online softmax ---------------------------------------
    const int kv0 = kv_start + t * BN;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < BN / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = kv0 + n * 8 + gc * 2 + (e & 1);
        const int pos = e < 2 ? pos0 : pos1;
        const int lo = e < 2 ? lo0 : lo1;
        const bool ok = j <= pos && j >= lo;
        const float v = s[n][e] * a.scale_log2 + slope * static_cast<float>(j - pos);
        s[n][e] = ok ? v : -INFINITY;
        if (e < 2) mx0 = fmaxf(mx0, s[n][e]); else mx1 = fmaxf(mx1, s[n][e]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;  // row with no key yet
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(m0 - mu0), al1 = fast_exp2(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int n = 0; n < BN / 8; ++n) {
      s[n][0] = fast_exp2(s[n][0] - mu0);
      s[n][1] = fast_exp2(s[n][1] - mu0);
      s[n][2] = fast_exp2(s[n][2] - mu1);
      s[n][3] = fast_exp2(s[n][3] - mu1);
      ps0 += s[n][0] + s[n][1];
      ps1 += s[n][2] + s[n][3];
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      oacc[n][0] *= al0;
      oacc[n][1] *= al0;
      oacc[n][2] *= al1;
      oacc[n][3] *= al1;
    }
    // ---- O += P V ----------------------------------------------------------
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = T::from_f2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = T::from_f2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = T::from_f2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = T::from_f2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int ndp = 0; ndp < D / 16; ++ndp) {
        const int key = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int c = ndp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz<D>(key, c), b0, b1, b2, b3);
        mma16816<T>(oacc[2 * ndp], pa, b0, b1);
        mma16816<T>(oacc[2 * ndp + 1], pa, b2, b3);
      }
    }
    __syncthreads();  // buffer `buf` is refilled two iterations later
  }

  // ---- epilogue -------------------------------------------------------------
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  uint16_t *out = static_cast<uint16_t *>(a.out);
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int d = n * 8 + gc * 2;
    if (r0 < q_rows) {
      uint32_t *p = reinterpret_cast<uint32_t *>(
          out + (static_cast<int64_t>(qs + q0 + r0) * a.H + h) * D + d);
      *p = T::from_f2(oacc[n][0] * inv0, oacc[n][1] * inv0);
    }
    if (r0 + 8 < q_rows) {
      uint32_t *p = reinterpret_cast<uint32_t *>(
          out + (static_cast<int64_t>(qs + q0 + r0 + 8) * a.H + h) * D + d);
      *p = T::from_f2(oacc[n][2] * inv1, oacc[n][3] * inv1);
    }
  }
}

template <class T, int D>
cudaError_t launch(const PrefillArgs &a, int max_query_len, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(BM) * D * 2 + 4ull * BN * D * 2;
  auto kern = prefill_mma_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tiles = (max_query_len + BM - 1) / BM;
  dim3 grid(a.H, a.num_seqs, tiles);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mma_path

// ===========================================================================
// tcgen05 / TMEM kernel (sm_100a family)
//
// CTA = (query head, sequence, 128-row query tile); 8 warps:
//   warp 0     TMA producer: the Q tile once, then per 128-key tile the K and
//              V rows of this KV head, one 4-D box (block_size rows x 64
//              dims, 128-byte swizzle) per cache block and 64-dim half,
//              straight from the paged cache through the block table; blocks
//              outside the visible range are loaded from an out-of-range
//              coordinate, which the TMA unit fills with zeros.
//   warp 1     MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//              score buffers (issued one tile ahead so the tensor core works
//              on S_{j+1} while the softmax warps work on S_j), then
//              O += P_j V_j with P_j read from TMEM (the "TS" form) and V_j
//              as an MN-major shared-memory operand.
//   warps 4-7  softmax: thread r owns TMEM lane r = query row r.  It loads
//              its 128 scores, applies scale, ALiBi and the causal / window
//              mask in the log2 domain, keeps a running max that is only
//              moved (and O rescaled in TMEM) when it grows by more than
//              2^8, writes P as bf16/fp16 pairs over the first 64 columns of
//              the score buffer, and finally normalises O and stores it.
//   warps 2-3  idle.
// TMEM: S0 = columns [0,128), S1 = [128,256), O = [256, 256 + head_size).
// Every wait is bounded; a timeout raises a CTA-wide abort flag, the roles
// stop, in-flight copies and MMAs are drained, TMEM is freed.
// ===========================================================================
namespace tc_path {

constexpr int BM = 128, BN = 128, NST = 2;
constexpr int kThreads = 256;

template <int D>
struct Lay {
  static constexpr int REG = 128 * 128;   // one 64-column region of 128 rows
  static constexpr int NREG = D / 64;
  static constexpr int TILE = REG * NREG;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_BAR = OFF_V + NST * TILE;
  static constexpr int B_Q = 0, B_KF = 1, B_VF = B_KF + NST, B_EMPTY = B_VF + NST,
                       B_SF = B_EMPTY + NST, B_PF = B_SF + 2, B_O = B_PF + 2, B_FIN = B_O + 1,
                       NBAR = B_FIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 32;
  // + alignment slack; at least ~114 KB so that one CTA owns an SM (and all
  // of its tensor memory)
  static constexpr int ALLOC = (BYTES + 1024) > 118 * 1024 ? (BYTES + 1024) : 118 * 1024;
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

template <class T, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
                  const __grid_constant__ CUtensorMap kvmap) {
  using L = Lay<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile uint32_t *abort_flag = misc + 1;

  const int h = blockIdx.x, b = blockIdx.y;
  const int tile = gridDim.z - 1 - blockIdx.z;
  TileSpan sp;
  if (!tile_span<BM, BN>(a, b, tile, threadIdx.x == 0 && h == 0, sp)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = h / a.QPK;
  const int BS = a.BS;
  const int TB = BN / BS;  // cache blocks per key tile
  const int ntiles = sp.ntiles;
  const int64_t where = static_cast<int64_t>(b) * a.H + h;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NBAR; ++i) mbar_init(&bars[i], i == L::B_PF || i == L::B_PF + 1 ? 128 : 1);
    misc[1] = 0;  // abort
    misc[2] = 0;  // key tiles issued
    fence_mbar_init();
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kvmap);
  }
  if (warp == 1) tc5::tmem_alloc<512>(misc);
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  const uint32_t tmem = misc[0];
  const uint32_t tmem_o = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int32_t *trow = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars[L::B_Q], L::TILE);
      for (int r = 0; r < L::NREG; ++r)
        tc5::tma_load_3d(smem + L::OFF_Q + r * L::REG, &qmap, &bars[L::B_Q], 64 * r, h,
                         sp.qs + sp.q0);
    }
    int j = 0;
    for (; j < ntiles; ++j) {
      const int s = j % NST;
      if (j >= NST && !warp_wait(&bars[L::B_EMPTY + s], ((j / NST) - 1) & 1, abort_flag, where))
        break;
      const int kv0 = sp.kv_start + j * BN;
      int coord = -BS;  // out of range: zero fill
      if (lane < TB) {
        const int lb = kv0 / BS + lane;
        const int p0 = lb * BS;
        if (p0 < sp.kv_end && p0 + BS > sp.kv_lo) {
          const int pb = __ldg(trow + lb);
          if (pb < 0 || pb >= a.num_blocks)
            record_error(PKV_ERR_BOUNDS, static_cast<int64_t>(b) * a.max_blocks_per_seq + lb);
          else
            coord = pb * BS;
        }
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[L::B_KF + s], L::TILE);
        mbar_arrive_expect_tx(&bars[L::B_VF + s], L::TILE);
      }
      __syncwarp();
      if (lane < TB) {
        uint8_t *kd = smem + L::OFF_K + s * L::TILE + lane * BS * 128;
        uint8_t *vd = smem + L::OFF_V + s * L::TILE + lane * BS * 128;
        for (int r = 0; r < L::NREG; ++r) {
          tma_load_4d(kd + r * L::REG, &kvmap, &bars[L::B_KF + s], 64 * r, g, coord, 0);
          tma_load_4d(vd + r * L::REG, &kvmap, &bars[L::B_VF + s], 64 * r, g, coord, 1);
        }
      }
    }
    if (lane == 0) misc[2] = static_cast<uint32_t>(j);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t ID_QK = tc5::idesc_f16(AB<T>::v, 0, BM, BN);
    constexpr uint32_t ID_PV = tc5::idesc_f16(AB<T>::v, 1, BM, D);
    bool ok = warp_wait(&bars[L::B_Q], 0, abort_flag, where);
    auto issue_qk = [&](int j) -> bool {
      const int s = j % NST;
      if (!warp_wait(&bars[L::B_KF + s], (j / NST) & 1, abort_flag, where)) return false;
      tc5::fence_after_sync();
      if (lane == 0) {
        const uint32_t sb = tmem + (j & 1) * 128;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const int r = k / 4, kk = k % 4;
          const uint64_t qd = tc5::sdesc_sw128(sbase + L::OFF_Q + r * L::REG + kk * 32, 16, 1024);
          const uint64_t kd =
              tc5::sdesc_sw128(sbase + L::OFF_K + s * L::TILE + r * L::REG + kk * 32, 16, 1024);
          tc5::mma_ss(sb, qd, kd, ID_QK, k > 0 ? 1u : 0u);
        }
        tc5::commit(&bars[L::B_SF + (j & 1)]);
      }
      __syncwarp();
      return true;
    };
    if (ok) ok = issue_qk(0);
    for (int j = 0; ok && j < ntiles; ++j) {
      if (j + 1 < ntiles && !issue_qk(j + 1)) break;
      const int s = j % NST;
      if (!warp_wait(&bars[L::B_VF + s], (j / NST) & 1, abort_flag, where)) break;
      // Positions past the sequence end hold whatever the cache holds there
      // (possibly non-finite); their P is exactly 0, but 0 * NaN is NaN, so
      // their V rows are zeroed before the PV product reads them.
      const int kv0 = sp.kv_start + j * BN;
      const int zr = max(0, sp.Lb - kv0);
      if (zr < BN) {
        uint8_t *vt = smem + L::OFF_V + s * L::TILE;
        const int n16 = (BN - zr) * 8;  // 16-byte chunks per region
        for (int r = 0; r < L::NREG; ++r)
          for (int c = lane; c < n16; c += 32)
            *reinterpret_cast<uint4 *>(vt + r * L::REG + zr * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (!warp_wait(&bars[L::B_PF + (j & 1)], (j >> 1) & 1, abort_flag, where)) break;
      tc5::fence_after_sync();
      if (lane == 0) {
        const uint32_t pb = tmem + (j & 1) * 128;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t vd =
              tc5::sdesc_sw128(sbase + L::OFF_V + s * L::TILE + k * 2048, L::REG, 1024);
          tc5::mma_ts(tmem_o, pb + k * 8, vd, ID_PV, (j > 0 || k > 0) ? 1u : 0u);
        }
        tc5::commit(&bars[L::B_EMPTY + s]);
        tc5::commit(&bars[L::B_O]);
      }
      __syncwarp();
    }
    // every MMA this thread issued has completed before TMEM is released
    if (lane == 0) tc5::commit(&bars[L::B_FIN]);
    __syncwarp();
    mbar_wait_bounded(&bars[L::B_FIN], 0, where);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int row = (warp - 4) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int pos = sp.cb + sp.q0 + row;
    const int lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
    const float slope = a.alibi ? __ldg(a.alibi + h) * kLog2e : 0.f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      if (!warp_wait(&bars[L::B_SF + (j & 1)], (j >> 1) & 1, abort_flag, where)) {
        ok = false;
        break;
      }
      tc5::fence_after_sync();
      const uint32_t sb = tmem + lane_base + (j & 1) * 128;
      uint32_t raw[BN / 32][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tc5::tmem_ld32(sb + 32 * c, raw[c]);
      tc5::tmem_ld_wait();
      const int kv0 = sp.kv_start + j * BN;
      const bool full = (kv0 + BN - 1 <= pos) && (kv0 >= lo);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int jj = kv0 + c * 32 + e;
          float x = fmaf(__uint_as_float(raw[c][e]), a.scale_log2,
                         slope * static_cast<float>(jj - pos));
          if (!full && (jj > pos || jj < lo)) x = -INFINITY;
          raw[c][e] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      // running max: moved only when it grows by more than 8 (2^8 in p)
      float alpha = 1.f;
      bool resc = false;
      if (m == -INFINITY) {
        m = mx;
      } else if (mx > m + 8.f) {
        alpha = fast_exp2(m - mx);
        m = mx;
        resc = true;
      }
      if (__any_sync(0xffffffffu, resc)) {
        // PV_{j-1} must have landed in O before it is rescaled
        if (!warp_wait(&bars[L::B_O], (j - 1) & 1, abort_flag, where)) {
          ok = false;
          break;
        }
        tc5::fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc5::tmem_ld32(tmem_o + lane_base + 32 * c, o);
          tc5::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc5::tmem_st32(tmem_o + lane_base + 32 * c, o);
        }
        tc5::tmem_st_wait();
      }
      l *= alpha;
      const float mu = m == -INFINITY ? 0.f : m;
      uint32_t pk[2][32];
      float ps = 0.f;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = fast_exp2(__uint_as_float(raw[c][e]) - mu);
          const float p1 = fast_exp2(__uint_as_float(raw[c][e + 1]) - mu);
          ps += p0 + p1;
          pk[(c * 32 + e) / 64][((c * 32 + e) % 64) / 2] = T::from_f2(p0, p1);
        }
      l += ps;
      tc5::tmem_st32(sb, pk[0]);
      tc5::tmem_st32(sb + 32, pk[1]);
      tc5::tmem_st_wait();
      tc5::fence_before_sync();
      mbar_arrive(&bars[L::B_PF + (j & 1)]);
    }
    if (ok && warp_wait(&bars[L::B_O], (ntiles - 1) & 1, abort_flag, where)) {
      tc5::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool valid = row < sp.q_rows;
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) +
                                             (static_cast<int64_t>(sp.qs + sp.q0 + row) * a.H + h) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc5::tmem_ld32(tmem_o + lane_base + 32 * c, o);
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
    const int issued = static_cast<int>(misc[2]);
    for (int s = 0; s < NST; ++s) {
      const int t_last = issued - 1 - ((issued - 1 - s) % NST + NST) % NST;
      if (t_last >= 0 && t_last % NST == s) {
        mbar_wait_bounded(&bars[L::B_KF + s], (t_last / NST) & 1, where);
        mbar_wait_bounded(&bars[L::B_VF + s], (t_last / NST) & 1, where);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc5::fence_after_sync();
    tc5::tmem_dealloc<512>(tmem);
  }
}

template <class T, int D>
cudaError_t launch(const PrefillArgs &a, int max_query_len, const CUtensorMap &qmap,
                   const CUtensorMap &kvmap, cudaStream_t stream) {
  const size_t smem = Lay<D>::ALLOC;
  auto kern = prefill_tc_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int tiles = (max_query_len + BM - 1) / BM;
  dim3 grid(a.H, a.num_seqs, tiles);
  kern<<<grid, kThreads, smem, stream>>>(a, qmap, kvmap);
  return cudaGetLastError();
}

}  // namespace tc_path

// ===========================================================================
// tcgen05 / TMEM kernel, two query tiles per CTA (ping-pong).
//
// CTA = two 128-row query tiles sharing every K/V tile: two query heads of one
// KV group on the same rows when the group has an even number of heads
// (grouped-query reuse), else the same head on two consecutive row tiles.
// 12 warps:
//   warp 0      TMA producer (the two Q tiles once; per 128-key tile the K and
//               V rows of the KV head, one box per cache block and 64-dim
//               half; blocks outside the visible range come from an
//               out-of-range coordinate, which the TMA unit zero-fills).
//   warp 1      MMA issuer (one thread), in the order
//                 QK_A(0) QK_B(0) | PV_A(j) QK_A(j+1) PV_B(j) QK_B(j+1) | ...
//               so the tensor core works on one tile while the other tile's
//               softmax runs.  S = Q K^T lands in the tile's TMEM score
//               buffer; O += P V reads P from TMEM (the "TS" form) and V as an
//               MN-major 128-byte-swizzled shared-memory operand.
//   warps 4-7   softmax of tile A, warps 8-11 of tile B: thread r owns TMEM
//               lane r = query row r; scores are loaded 128 at a time, masked
//               (causal, window, range) only on tiles that need it, the
//               running max is moved (and O rescaled in TMEM) only when it
//               grows by more than 2^8, and P is written back as bf16/fp16
//               pairs over the first 64 columns of the score buffer, 16
//               columns at a time.
//   warps 2-3   idle.
// TMEM: S_A [0,128), S_B [128,256), O_A [256, 256+D), O_B [384, 384+D).
// Every wait is bounded; a timeout raises a CTA-wide abort flag, the roles
// stop, in-flight copies and MMAs are drained, TMEM is freed.
// ===========================================================================
namespace tc2 {

constexpr int BM = 128, BN = 128, NST = 2;
constexpr int kThreads = 384;

template <int D>
struct Lay {
  static constexpr int REG = 128 * 128;
  static constexpr int NREG = D / 64;
  static constexpr int TILE = REG * NREG;
  static constexpr int OFF_Q = 0;  // two Q tiles
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_BAR = OFF_V + NST * TILE;
  static constexpr int B_Q = 0, B_KF = 1, B_VF = B_KF + NST, B_EMPTY = B_VF + NST,
                       B_SF = B_EMPTY + NST, B_PF = B_SF + 2, B_O = B_PF + 2, B_FIN = B_O + 2,
                       NBAR = B_FIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 32;
  static constexpr int ALLOC = (BYTES + 1024) > 118 * 1024 ? (BYTES + 1024) : 118 * 1024;
};

// One query tile of the CTA: head, first row within the sequence, rows,
// and the half-open range of the CTA's key tiles it needs.
struct QTile {
  int head, q0, rows, j0, j1;
};

template <class T, int D, bool ALIBI>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc2_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kvmap, int pair_heads) {
  using L = Lay<D>;
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
      end_t[x] = i_last + 1;
      kv_lo = min(kv_lo, lo_t[x]);
      kv_end = max(kv_end, end_t[x]);
    }
  }
  const int kv_start = kv_lo / BN * BN;
  const int ntiles = (kv_end - kv_start + BN - 1) / BN;
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
    for (int i = 0; i < L::NBAR; ++i)
      mbar_init(&bars[i], (i == L::B_PF || i == L::B_PF + 1) ? 128 : 1);
    misc[1] = 0;
    misc[2] = 0;
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
    int j = 0;
    for (; j < ntiles; ++j) {
      const int s = j % NST;
      if (j >= NST && !tc_path::warp_wait(&bars[L::B_EMPTY + s], ((j / NST) - 1) & 1, abort_flag,
                                          where))
        break;
      const int kv0 = kv_start + j * BN;
      int coord = -BS;  // out of range: zero fill
      if (lane < TB) {
        const int lb = kv0 / BS + lane;
        const int p0 = lb * BS;
        if (p0 < kv_end && p0 + BS > kv_lo) {
          const int pb = __ldg(trow + lb);
          if (pb < 0 || pb >= a.num_blocks)
            record_error(PKV_ERR_BOUNDS, static_cast<int64_t>(b) * a.max_blocks_per_seq + lb);
          else
            coord = pb * BS;
        }
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[L::B_KF + s], L::TILE);
        mbar_arrive_expect_tx(&bars[L::B_VF + s], L::TILE);
      }
      __syncwarp();
      if (lane < TB) {
        uint8_t *kd = smem + L::OFF_K + s * L::TILE + lane * BS * 128;
        uint8_t *vd = smem + L::OFF_V + s * L::TILE + lane * BS * 128;
        for (int r = 0; r < L::NREG; ++r) {
          tma_load_4d(kd + r * L::REG, &kvmap, &bars[L::B_KF + s], 64 * r, g, coord, 0);
          tma_load_4d(vd + r * L::REG, &kvmap, &bars[L::B_VF + s], 64 * r, g, coord, 1);
        }
      }
    }
    if (lane == 0) misc[2] = static_cast<uint32_t>(j);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t ID_QK = tc5::idesc_f16(tc_path::AB<T>::v, 0, BM, BN);
    constexpr uint32_t ID_PV = tc5::idesc_f16(tc_path::AB<T>::v, 1, BM, D);
    bool ok = tc_path::warp_wait(&bars[L::B_Q], 0, abort_flag, where);
    int k_ready = -1;  // highest key tile known to have landed
    auto need_k = [&](int j) -> bool {
      if (j <= k_ready) return true;
      if (!tc_path::warp_wait(&bars[L::B_KF + j % NST], (j / NST) & 1, abort_flag, where))
        return false;
      tc5::fence_after_sync();
      k_ready = j;
      return true;
    };
    auto qk = [&](int x, int j) {
      if (lane == 0) {
        const int s = j % NST;
        const uint32_t sb = tmem + x * 128;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const int r = k / 4, kk = k % 4;
          const uint64_t qd =
              tc5::sdesc_sw128(sbase + L::OFF_Q + x * L::TILE + r * L::REG + kk * 32, 16, 1024);
          const uint64_t kd =
              tc5::sdesc_sw128(sbase + L::OFF_K + s * L::TILE + r * L::REG + kk * 32, 16, 1024);
          tc5::mma_ss(sb, qd, kd, ID_QK, k > 0 ? 1u : 0u);
        }
        tc5::commit(&bars[L::B_SF + x]);
      }
      __syncwarp();
    };
    const int j0A = qt[0].j0, j1A = qt[0].j1, j0B = qt[1].j0, j1B = qt[1].j1;
    auto active = [&](int x, int j) {
      return x == 0 ? (j >= j0A && j < j1A) : (j >= j0B && j < j1B);
    };
    if (ok && ntiles > 0) {
      ok = need_k(0);
      if (ok) {
        if (active(0, 0)) qk(0, 0);
        if (active(1, 0)) qk(1, 0);
      }
    }
    int pf_a = 0, pf_b = 0;  // P tiles consumed per query tile
    // PV of tile x for key tile j, then the look-ahead QK of tile x
    auto step = [&](int x, int j, int s, int &pf) -> bool {
      if (active(x, j)) {
        if (!tc_path::warp_wait(&bars[L::B_PF + x], pf & 1, abort_flag, where)) return false;
        tc5::fence_after_sync();
        if (lane == 0) {
          const uint32_t pb = tmem + x * 128;
          const uint32_t ob = tmem + 256 + x * 128;
#pragma unroll
          for (int k = 0; k < BN / 16; ++k) {
            const uint64_t vd =
                tc5::sdesc_sw128(sbase + L::OFF_V + s * L::TILE + k * 2048, L::REG, 1024);
            tc5::mma_ts(ob, pb + k * 8, vd, ID_PV, (pf > 0 || k > 0) ? 1u : 0u);
          }
          tc5::commit(&bars[L::B_O + x]);
        }
        __syncwarp();
        ++pf;
      }
      if (j + 1 < ntiles && active(x, j + 1)) {
        if (!need_k(j + 1)) return false;
        qk(x, j + 1);
      }
      return true;
    };
    for (int j = 0; ok && j < ntiles; ++j) {
      const int s = j % NST;
      if (!tc_path::warp_wait(&bars[L::B_VF + s], (j / NST) & 1, abort_flag, where)) break;
      // rows past the sequence end: P there is exactly 0, but the cache may
      // hold non-finite values and 0 * NaN is NaN, so zero those V rows
      const int kv0 = kv_start + j * BN;
      const int zr = max(0, Lb - kv0);
      if (zr < BN) {
        uint8_t *vt = smem + L::OFF_V + s * L::TILE;
        const int n16 = (BN - zr) * 8;
        for (int r = 0; r < L::NREG; ++r)
          for (int c = lane; c < n16; c += 32)
            *reinterpret_cast<uint4 *>(vt + r * L::REG + zr * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (!step(0, j, s, pf_a) || !step(1, j, s, pf_b)) break;
      if (lane == 0) tc5::commit(&bars[L::B_EMPTY + s]);
      __syncwarp();
    }
    if (lane == 0) tc5::commit(&bars[L::B_FIN]);
    __syncwarp();
    mbar_wait_bounded(&bars[L::B_FIN], 0, where);
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
    const float sl2 = a.scale_log2;
    const float slope = ALIBI ? __ldg(a.alibi + t.head) * kLog2e : 0.f;
    // running max m: in the log2 domain with ALiBi; in raw-score units
    // without (then scores are scaled inside the exponent's FMA)
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    const int n = t.j1 - t.j0;
    for (int k = 0; k < n; ++k) {
      const int j = t.j0 + k;
      if (!tc_path::warp_wait(&bars[L::B_SF + x], k & 1, abort_flag, where)) {
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
      const bool full = (kv0 + BN - 1 <= pos) && (kv0 >= lo);
      float mx = -INFINITY;
      if constexpr (ALIBI) {
        const float b0 = slope * static_cast<float>(kv0 - pos);
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          float v = fmaf(__uint_as_float(raw[e]), sl2, fmaf(slope, static_cast<float>(e), b0));
          if (!full && (kv0 + e > pos || kv0 + e < lo)) v = -INFINITY;
          raw[e] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      } else {
        if (!full) {
#pragma unroll
          for (int e = 0; e < BN; ++e)
            if (kv0 + e > pos || kv0 + e < lo) raw[e] = __float_as_uint(-INFINITY);
        }
#pragma unroll
        for (int e = 0; e < BN; ++e) mx = fmaxf(mx, __uint_as_float(raw[e]));
      }
      // move the max only when it grows by more than 8 (2^8 in p)
      float alpha = 1.f;
      bool resc = false;
      const float unit = ALIBI ? 1.f : sl2;  // log2 units per unit of m
      if (m == -INFINITY) {
        m = mx;
      } else if ((mx - m) * unit > 8.f) {
        alpha = fast_exp2((m - mx) * unit);
        m = mx;
        resc = true;
      }
      const float mu = m == -INFINITY ? 0.f : m * unit;
      float ps = 0.f;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p0, p1;
          if constexpr (ALIBI) {
            p0 = fast_exp2(__uint_as_float(raw[32 * c + e]) - mu);
            p1 = fast_exp2(__uint_as_float(raw[32 * c + e + 1]) - mu);
          } else {
            p0 = fast_exp2(fmaf(__uint_as_float(raw[32 * c + e]), sl2, -mu));
            p1 = fast_exp2(fmaf(__uint_as_float(raw[32 * c + e + 1]), sl2, -mu));
          }
          ps += p0 + p1;
          pk[e / 2] = T::from_f2(p0, p1);
        }
        tc5::tmem_st16(sb + 16 * c, pk);
      }
      l = l * alpha + ps;
      if (__any_sync(0xffffffffu, resc)) {
        // O_x holds PV of the previous key tile once it has completed
        if (!tc_path::warp_wait(&bars[L::B_O + x], (k - 1) & 1, abort_flag, where)) {
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
    if (ok && n > 0 && tc_path::warp_wait(&bars[L::B_O + x], (n - 1) & 1, abort_flag, where)) {
      tc5::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
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
    mbar_wait_bounded(&bars[L::B_Q], 0, where);
    const int issued = static_cast<int>(misc[2]);
    for (int s = 0; s < NST; ++s) {
      const int t_last = issued - 1 - ((issued - 1 - s) % NST + NST) % NST;
      if (t_last >= 0 && t_last % NST == s) {
        mbar_wait_bounded(&bars[L::B_KF + s], (t_last / NST) & 1, where);
        mbar_wait_bounded(&bars[L::B_VF + s], (t_last / NST) & 1, where);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc5::fence_after_sync();
    tc5::tmem_dealloc<512>(tmem);
  }
}

template <class T, int D, bool ALIBI>
cudaError_t launch(const PrefillArgs &a, int max_query_len, const CUtensorMap &qmap,
                   const CUtensorMap &kvmap, cudaStream_t stream) {
  const size_t smem = Lay<D>::ALLOC;
  auto kern = prefill_tc2_kernel<T, D, ALIBI>;
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
                       const CUtensorMap &kvmap, cudaStream_t stream) {
  return a.alibi ? launch<T, D, true>(a, max_query_len, qmap, kvmap, stream)
                 : launch<T, D, false>(a, max_query_len, qmap, kvmap, stream);
}

}  // namespace tc2

cudaError_t launch_prefill(void *out, const void *query, int64_t num_q_tokens, int num_seqs,
                           const int32_t *cu_q, const int32_t *cu_k, int max_query_len,
                           int max_seq_len, const void *kv_cache, const int32_t *block_tables,
                           int max_blocks_per_seq, const Geometry &g, cudaStream_t stream) {
  (void)max_seq_len;
  PrefillArgs a{};
  a.out = out;
  a.query = static_cast<const uint16_t *>(query);
  a.k_half = static_cast<const uint16_t *>(kv_cache);
  a.v_half = a.k_half + g.num_blocks * g.block_elems;
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
  a.scale_log2 = g.scale * kLog2e;
  const bool bf = g.dtype == PKV_BF16;
#ifdef PKV_PREFILL_MMA_SYNC
  if (g.D == 128) return bf ? mma_path::launch<BF16, 128>(a, max_query_len, stream)
                            : mma_path::launch<FP16, 128>(a, max_query_len, stream);
  if (g.D == 64) return bf ? mma_path::launch<BF16, 64>(a, max_query_len, stream)
                           : mma_path::launch<FP16, 64>(a, max_query_len, stream);
  return cudaErrorInvalidValue;
#else
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
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(tc_path::BM)};
    if (encode_tensor_map(&qmap, dt, 3, const_cast<void *>(query), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(g.D), static_cast<cuuint64_t>(g.KVH),
                                static_cast<cuuint64_t>(g.num_blocks * g.BS), 2};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(g.D) * 2,
                                   static_cast<cuuint64_t>(g.row_elems) * 2,
                                   static_cast<cuuint64_t>(g.num_blocks * g.block_elems) * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(g.BS), 1};
    if (encode_tensor_map(&kvmap, dt, 4, const_cast<void *>(kv_cache), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
#ifdef PKV_PREFILL_TC1
  if (g.D == 128) return bf ? tc_path::launch<BF16, 128>(a, max_query_len, qmap, kvmap, stream)
                            : tc_path::launch<FP16, 128>(a, max_query_len, qmap, kvmap, stream);
  if (g.D == 64) return bf ? tc_path::launch<BF16, 64>(a, max_query_len, qmap, kvmap, stream)
                           : tc_path::launch<FP16, 64>(a, max_query_len, qmap, kvmap, stream);
#else
  if (g.D == 128) return bf ? tc2::launch_any<BF16, 128>(a, max_query_len, qmap, kvmap, stream)
                            : tc2::launch_any<FP16, 128>(a, max_query_len, qmap, kvmap, stream);
  if (g.D == 64) return bf ? tc2::launch_any<BF16, 64>(a, max_query_len, qmap, kvmap, stream)
                           : tc2::launch_any<FP16, 64>(a, max_query_len, qmap, kvmap, stream);
#endif
  return cudaErrorInvalidValue;
#endif
}

cudaError_t read_device_error_prefill(unsigned long long *out) {
  return read_and_clear_unit_error(out);
}

}  // namespace pkv
