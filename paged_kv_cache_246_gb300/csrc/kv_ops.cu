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
// kv_cache_write: warp w of the grid copies tokens w, w + warps, ...: its
// lanes take the row's 16-byte chunks lane, lane + 32, ..., U of them in
// flight per lane for each half; the slot is read once per token.  No
// per-chunk index arithmetic beyond an add.
// ---------------------------------------------------------------------------
constexpr int kWriteThreads = 256;
constexpr int kWriteWarps = kWriteThreads / 32;

template <int U>
__global__ void __launch_bounds__(kWriteThreads)
kv_write_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value, int64_t num_tokens,
                uint4 *__restrict__ k_half, uint4 *__restrict__ v_half,
                const int64_t *__restrict__ slots, int64_t num_slots, int row_chunks) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kWriteWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWriteWarps + (threadIdx.x >> 5);
       t < num_tokens; t += warps) {
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;  // padding token
    if (s >= num_slots) {
      if (lane == 0) record_error(PKV_ERR_BOUNDS, t);
      continue;
    }
    const uint4 *kr = key + t * row_chunks, *vr = value + t * row_chunks;
    uint4 *kd = k_half + s * row_chunks, *vd = v_half + s * row_chunks;
    int c = lane;
    for (; c + 32 * (U - 1) < row_chunks; c += 32 * U) {
      uint4 kk[U], vv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        kk[u] = __ldg(kr + c + 32 * u);
        vv[u] = __ldg(vr + c + 32 * u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        kd[c + 32 * u] = kk[u];
        vd[c + 32 * u] = vv[u];
      }
    }
    for (; c < row_chunks; c += 32) {
      kd[c] = __ldg(kr + c);
      vd[c] = __ldg(vr + c);
    }
  }
}

// fp8 cache: lane chunk c of a token is 16 codes, made from 16 input
// elements (two 16-byte input chunks): code = nearest E4M3 to x / scale
// (IEEE fp32 division, round to nearest even, saturating at 448).
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
__device__ __forceinline__ uint4 quant16(uint4 a, uint4 b, float scale) {
  return make_uint4(quant4<T>(make_uint2(a.x, a.y), scale), quant4<T>(make_uint2(a.z, a.w), scale),
                    quant4<T>(make_uint2(b.x, b.y), scale), quant4<T>(make_uint2(b.z, b.w), scale));
}

template <class T>
__global__ void __launch_bounds__(kWriteThreads)
kv_write_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                    int64_t num_tokens, uint4 *__restrict__ k_half, uint4 *__restrict__ v_half,
                    const int64_t *__restrict__ slots, int64_t num_slots, int row_chunks,
                    float k_scale, float v_scale) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kWriteWarps;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWriteWarps + (threadIdx.x >> 5);
       t < num_tokens; t += warps) {
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;  // padding token
    if (s >= num_slots) {
      if (lane == 0) record_error(PKV_ERR_BOUNDS, t);
      continue;
    }
    const uint4 *kr = key + 2 * t * row_chunks, *vr = value + 2 * t * row_chunks;
    uint4 *kd = k_half + s * row_chunks, *vd = v_half + s * row_chunks;
    for (int c = lane; c < row_chunks; c += 32) {
      const uint4 k0 = __ldg(kr + 2 * c), k1 = __ldg(kr + 2 * c + 1);
      const uint4 v0 = __ldg(vr + 2 * c), v1 = __ldg(vr + 2 * c + 1);
      kd[c] = quant16<T>(k0, k1, k_scale);
      vd[c] = quant16<T>(v0, v1, v_scale);
    }
  }
}

cudaError_t launch_kv_write(const void *key, const void *value, int64_t num_tokens, void *kv_cache,
                            const int64_t *slot_mapping, const Geometry &g, cudaStream_t stream) {
  DeviceInfo dev;
  cudaError_t e = current_device_info(&dev);
  if (e != cudaSuccess) return e;
  const int row_chunks = static_cast<int>(g.row_bytes / 16);  // 16-byte chunks of a cache row
  const int64_t num_slots = g.num_blocks * g.BS;
  uint4 *k_half = static_cast<uint4 *>(kv_cache);
  uint4 *v_half = k_half + num_slots * row_chunks;
  // one warp per token, up to 8 CTAs per SM
  const int blocks = static_cast<int>(std::min<int64_t>(
      (num_tokens + kWriteWarps - 1) / kWriteWarps, int64_t(dev.sms) * 8));
  const uint4 *k = static_cast<const uint4 *>(key), *v = static_cast<const uint4 *>(value);
  if (g.fp8) {
    auto kern = g.dtype == PKV_BF16 ? kv_write_fp8_kernel<BF16> : kv_write_fp8_kernel<FP16>;
    kern<<<blocks, kWriteThreads, 0, stream>>>(k, v, num_tokens, k_half, v_half, slot_mapping,
                                               num_slots, row_chunks, g.k_scale, g.v_scale);
  } else {
    kv_write_kernel<4><<<blocks, kWriteThreads, 0, stream>>>(k, v, num_tokens, k_half, v_half,
                                                             slot_mapping, num_slots, row_chunks);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// kv_copy_blocks: CTA (piece, pair, layer) copies piece `piece` (16 KiB, or
// the rest) of both halves of one block: 256 threads x kCopyUnroll 16-byte
// chunks in flight per half.  Short CTAs keep the tail of the grid short.
// ---------------------------------------------------------------------------
constexpr int kMaxLayers = 256;
struct LayerPtrs {
  uint4 *p[kMaxLayers];
};
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kCopyPieceChunks = kCopyThreads * kCopyUnroll;  // 16 KiB

__global__ void __launch_bounds__(kCopyThreads)
kv_copy_kernel(const __grid_constant__ LayerPtrs caches, const int64_t *__restrict__ pairs,
               int64_t first_pair, int64_t num_blocks, int64_t block_chunks) {
  const int64_t pair = first_pair + blockIdx.y;
  const int layer = blockIdx.z;
  const int64_t s = __ldg(pairs + 2 * pair);
  const int64_t d = __ldg(pairs + 2 * pair + 1);
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(PKV_ERR_BOUNDS, pair);
    return;
  }
  const int64_t half = num_blocks * block_chunks;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kCopyPieceChunks + threadIdx.x;
  const uint4 *src = caches.p[layer] + s * block_chunks;
  uint4 *dst = caches.p[layer] + d * block_chunks;
  uint4 r[2][kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t c = c0 + u * kCopyThreads;
    if (c < block_chunks) {
      r[0][u] = src[c];
      r[1][u] = src[half + c];
    }
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t c = c0 + u * kCopyThreads;
    if (c < block_chunks) {
      dst[c] = r[0][u];
      dst[half + c] = r[1][u];
    }
  }
}

cudaError_t launch_kv_copy(void *const *caches, int num_layers, const int64_t *pairs,
                           int64_t num_pairs, const Geometry &g, cudaStream_t stream) {
  LayerPtrs lp;
  for (int l = 0; l < kMaxLayers; ++l)
    lp.p[l] = l < num_layers ? static_cast<uint4 *>(caches[l]) : nullptr;
  const int64_t block_chunks = g.block_bytes / 16;
  const unsigned pieces = static_cast<unsigned>((block_chunks + kCopyPieceChunks - 1) / kCopyPieceChunks);
  // grid.y may go up to 65535: pairs beyond that are split over launches
  const int64_t max_y = 65535;
  for (int64_t a = 0; a < num_pairs; a += max_y) {
    const int64_t n = std::min(max_y, num_pairs - a);
    dim3 grid(pieces, static_cast<unsigned>(n), num_layers);
    kv_copy_kernel<<<grid, kCopyThreads, 0, stream>>>(lp, pairs, a, g.num_blocks, block_chunks);
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
