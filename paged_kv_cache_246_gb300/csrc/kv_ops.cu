// Bandwidth kernels: the cache write (reshape_and_cache) and the block moves
// (copy_blocks, swap_blocks) of the xformers.py / cpu_attn backends.
//
// All three are pure 16-byte vector copies.  Rows (KVH * D elements) and
// blocks (BS * KVH * D elements) are multiples of 16 bytes for every
// supported head size, so every access is an aligned uint4.
#include <cuda_fp8.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// kv_cache_write: thread i copies 16-byte chunk (i % row_chunks) of token
// (i / row_chunks) into K and V halves at its slot.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
kv_write_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value, int64_t num_tokens,
                uint4 *__restrict__ k_half, uint4 *__restrict__ v_half,
                const int64_t *__restrict__ slots, int64_t num_slots, int row_chunks) {
  const int64_t total = num_tokens * row_chunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / row_chunks;
    const int64_t c = i - t * row_chunks;
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;  // padding token
    if (s >= num_slots) {
      record_error(PKV_ERR_BOUNDS, t);
      continue;
    }
    const uint4 kv = __ldg(key + i);
    const uint4 vv = __ldg(value + i);
    k_half[s * row_chunks + c] = kv;
    v_half[s * row_chunks + c] = vv;
  }
}

// fp8 cache: thread i produces 16-byte chunk (i % row_chunks) of codes of
// token (i / row_chunks), from 16 input elements: code = nearest E4M3 to
// x / scale (IEEE fp32 division, round to nearest even, saturating at 448).
template <class T>
__device__ __forceinline__ uint32_t quant4(uint2 in, float scale) {
  float2 a = T::to_f2(in.x), b = T::to_f2(in.y);
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
      make_float2(__fdiv_rn(a.x, scale), __fdiv_rn(a.y, scale)), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
      make_float2(__fdiv_rn(b.x, scale), __fdiv_rn(b.y, scale)), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

template <class T>
__global__ void __launch_bounds__(256)
kv_write_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                    int64_t num_tokens, uint4 *__restrict__ k_half, uint4 *__restrict__ v_half,
                    const int64_t *__restrict__ slots, int64_t num_slots, int row_chunks,
                    float k_scale, float v_scale) {
  const int64_t total = num_tokens * row_chunks;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / row_chunks;
    const int64_t c = i - t * row_chunks;
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;  // padding token
    if (s >= num_slots) {
      record_error(PKV_ERR_BOUNDS, t);
      continue;
    }
    const uint4 k0 = __ldg(key + 2 * i), k1 = __ldg(key + 2 * i + 1);
    const uint4 v0 = __ldg(value + 2 * i), v1 = __ldg(value + 2 * i + 1);
    k_half[s * row_chunks + c] =
        make_uint4(quant4<T>(make_uint2(k0.x, k0.y), k_scale), quant4<T>(make_uint2(k0.z, k0.w), k_scale),
                   quant4<T>(make_uint2(k1.x, k1.y), k_scale), quant4<T>(make_uint2(k1.z, k1.w), k_scale));
    v_half[s * row_chunks + c] =
        make_uint4(quant4<T>(make_uint2(v0.x, v0.y), v_scale), quant4<T>(make_uint2(v0.z, v0.w), v_scale),
                   quant4<T>(make_uint2(v1.x, v1.y), v_scale), quant4<T>(make_uint2(v1.z, v1.w), v_scale));
  }
}

cudaError_t launch_kv_write(const void *key, const void *value, int64_t num_tokens, void *kv_cache,
                            const int64_t *slot_mapping, const Geometry &g, cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t e = current_device_info(&dev);
  if (e != cudaSuccess) return e;
  if (g.fp8) {
    const int row_chunks = static_cast<int>(g.row_bytes / 16);  // 16 codes per chunk
    const int64_t num_slots = g.num_blocks * g.BS;
    uint4 *k_half = static_cast<uint4 *>(kv_cache);
    uint4 *v_half = k_half + num_slots * row_chunks;
    const int64_t total = num_tokens * row_chunks;
    const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, int64_t(dev.sms) * 8));
    auto kern = g.dtype == PKV_BF16 ? kv_write_fp8_kernel<BF16> : kv_write_fp8_kernel<FP16>;
    kern<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(key),
                                     static_cast<const uint4 *>(value), num_tokens, k_half, v_half,
                                     slot_mapping, num_slots, row_chunks, g.k_scale, g.v_scale);
    return cudaGetLastError();
  }
  const int row_chunks = static_cast<int>(g.row_elems * 2 / 16);
  const int64_t num_slots = g.num_blocks * g.BS;
  uint4 *k_half = static_cast<uint4 *>(kv_cache);
  uint4 *v_half = k_half + num_slots * row_chunks;
  const int64_t total = num_tokens * row_chunks;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(std::min<int64_t>(want, int64_t(dev.sms) * 8));
  kv_write_kernel<<<blocks, threads, 0, stream>>>(
      static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), num_tokens, k_half,
      v_half, slot_mapping, num_slots, row_chunks);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// kv_copy_blocks: CTA (pair, layer) copies one block in both halves.
// ---------------------------------------------------------------------------
constexpr int kMaxLayers = 256;
struct LayerPtrs {
  uint4 *p[kMaxLayers];
};

template <int UNROLL>
__device__ __forceinline__ void copy_chunks(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                            int64_t n) {
  int64_t c = threadIdx.x;
  for (; c + (UNROLL - 1) * static_cast<int64_t>(blockDim.x) < n; c += UNROLL * blockDim.x) {
    uint4 r[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) r[u] = src[c + u * blockDim.x];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) dst[c + u * blockDim.x] = r[u];
  }
  for (; c < n; c += blockDim.x) dst[c] = src[c];
}

__global__ void __launch_bounds__(256)
kv_copy_kernel(const __grid_constant__ LayerPtrs caches, const int64_t *__restrict__ pairs,
               int64_t num_blocks, int64_t block_chunks) {
  const int64_t pair = blockIdx.x;
  const int layer = blockIdx.y;
  const int64_t s = __ldg(pairs + 2 * pair);
  const int64_t d = __ldg(pairs + 2 * pair + 1);
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0) record_error(PKV_ERR_BOUNDS, pair);
    return;
  }
  uint4 *base = caches.p[layer];
  const int64_t half = num_blocks * block_chunks;
  copy_chunks<4>(base + d * block_chunks, base + s * block_chunks, block_chunks);
  copy_chunks<4>(base + half + d * block_chunks, base + half + s * block_chunks, block_chunks);
}

cudaError_t launch_kv_copy(void *const *caches, int num_layers, const int64_t *pairs,
                           int64_t num_pairs, const Geometry &g, cudaStream_t stream) {
  LayerPtrs lp;
  for (int l = 0; l < kMaxLayers; ++l)
    lp.p[l] = l < num_layers ? static_cast<uint4 *>(caches[l]) : nullptr;
  const int64_t block_chunks = g.block_bytes / 16;
  // grid.x may go up to 2^31-1: pairs beyond that are split over launches
  const int64_t max_x = 0x7fffffff;
  for (int64_t a = 0; a < num_pairs; a += max_x) {
    const int64_t n = std::min(max_x, num_pairs - a);
    dim3 grid(static_cast<unsigned>(n), num_layers);
    kv_copy_kernel<<<grid, 256, 0, stream>>>(lp, pairs + 2 * a, g.num_blocks, block_chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// kv_swap_blocks: the pair list is host memory, so it travels in the kernel's
// parameter space (kSwapChunk pairs per launch, already range-checked on
// the host).  CTA (k, half) moves block src[k] -> dst[k] of that half.
// One side is normally pinned host memory reached over the chip-to-host
// link; the many outstanding 16-byte requests of 256 threads x UNROLL keep
// the link busy.
// ---------------------------------------------------------------------------
constexpr int kSwapChunk = 1536;
struct SwapPairs {
  int32_t src[kSwapChunk];
  int32_t dst[kSwapChunk];
};

__global__ void __launch_bounds__(256)
kv_swap_kernel(const uint4 *__restrict__ src, int64_t src_half, uint4 *__restrict__ dst,
               int64_t dst_half, const __grid_constant__ SwapPairs pp, int64_t block_chunks) {
  const int k = blockIdx.x;
  const int half = blockIdx.y;
  const int64_t s = pp.src[k];
  const int64_t d = pp.dst[k];
  copy_chunks<8>(dst + half * dst_half + d * block_chunks, src + half * src_half + s * block_chunks,
                 block_chunks);
}

cudaError_t launch_kv_swap(const void *src, int64_t src_blocks, void *dst, int64_t dst_blocks,
                           const int64_t *pairs_host, int64_t num_pairs, const Geometry &g,
                           cudaStream_t stream) {
  const int64_t block_chunks = g.block_bytes / 16;
  SwapPairs pp;
  for (int64_t a = 0; a < num_pairs; a += kSwapChunk) {
    const int n = static_cast<int>(std::min<int64_t>(kSwapChunk, num_pairs - a));
    for (int k = 0; k < n; ++k) {
      pp.src[k] = static_cast<int32_t>(pairs_host[2 * (a + k)]);
      pp.dst[k] = static_cast<int32_t>(pairs_host[2 * (a + k) + 1]);
    }
    kv_swap_kernel<<<dim3(n, 2), 256, 0, stream>>>(
        static_cast<const uint4 *>(src), src_blocks * block_chunks, static_cast<uint4 *>(dst),
        dst_blocks * block_chunks, pp, block_chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// A wait on an mbarrier that nothing will complete, bounded like every wait
// of the library: it gives up after kWaitLimitNs, records PKV_ERR_TIMEOUT with
// `tag` and returns; nothing else is in flight, so the CTA simply ends.
__global__ void wait_timeout_check_kernel(int64_t tag) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait_bounded(&bar, 0, tag);
  }
}

cudaError_t launch_wait_timeout_check(int64_t tag, cudaStream_t stream) {
  wait_timeout_check_kernel<<<1, 32, 0, stream>>>(tag);
  return cudaGetLastError();
}

cudaError_t read_device_error_kv_ops(unsigned long long *out) {
  return read_and_clear_unit_error(out);
}

}  // namespace pkv
