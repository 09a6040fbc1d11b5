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
  int num_seqs, max_blocks_per_seq;
  int H, KVH, QPK, BS, window;
  float scale_log2;
};

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
  const int q0 = tile * BM;
  const int qs = __ldg(a.cu_q + b), qb = __ldg(a.cu_q + b + 1) - qs;
  const int Lb = __ldg(a.cu_k + b + 1) - __ldg(a.cu_k + b);
  if (q0 >= qb) return;
  const bool report = (threadIdx.x == 0 && h == 0);
  if (qb > Lb || Lb > a.max_blocks_per_seq * a.BS) {
    if (report) record_error(PKV_ERR_BOUNDS, b);
    return;
  }
  const int cb = Lb - qb;
  const int g = h / a.QPK;
  const int q_rows = min(BM, qb - q0);
  const int i_first = cb + q0, i_last = cb + q0 + q_rows - 1;
  const int kv_lo = a.window > 0 ? max(0, i_first - a.window + 1) : 0;
  const int kv_start = kv_lo / BN * BN;
  const int kv_end = i_last + 1;  // exclusive
  const int ntiles = (kv_end - kv_start + BN - 1) / BN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t *trow = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
  const int64_t kv_row_stride = static_cast<int64_t>(a.KVH) * D;

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
  (void)kv_row_stride;

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

cudaError_t launch_prefill(void *out, const void *query, int num_seqs, const int32_t *cu_q,
                           const int32_t *cu_k, int max_query_len, int max_seq_len,
                           const void *kv_cache, const int32_t *block_tables,
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
  a.num_seqs = num_seqs;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.H = g.H;
  a.KVH = g.KVH;
  a.QPK = g.QPK;
  a.BS = g.BS;
  a.window = g.window;
  a.scale_log2 = g.scale * kLog2e;
  const bool bf = g.dtype == PKV_BF16;
  if (g.D == 128) return bf ? mma_path::launch<BF16, 128>(a, max_query_len, stream)
                            : mma_path::launch<FP16, 128>(a, max_query_len, stream);
  if (g.D == 64) return bf ? mma_path::launch<BF16, 64>(a, max_query_len, stream)
                           : mma_path::launch<FP16, 64>(a, max_query_len, stream);
  return cudaErrorInvalidValue;
}

cudaError_t read_device_error_prefill(unsigned long long *out) {
  return read_and_clear_unit_error(out);
}

}  // namespace pkv
