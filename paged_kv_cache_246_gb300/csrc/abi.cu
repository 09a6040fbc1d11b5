// extern "C" front end of libpkv.so: argument validation, device selection
// and dispatch to the kernels of kv_ops.cu, decode.cu and prefill.cu.
// Everything here runs on the host; nothing reads device memory.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Device facts, cached per device
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
static DeviceInfo g_dev_info[kMaxDevices];
static bool g_dev_known[kMaxDevices];
static std::mutex g_mu;

cudaError_t current_device_info(DeviceInfo *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev_known[dev]) {
    DeviceInfo d{dev, 0, 0};
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    g_dev_info[dev] = d;
    g_dev_known[dev] = true;
  }
  *out = g_dev_info[dev];
  return cudaSuccess;
}

// The library runs on the device that owns the caller's stream and leaves
// the calling thread's current device as it found it: a DeviceScope makes the
// stream's device current for the launches of one call and restores the
// previous device when the call returns.  The legacy and per-thread default
// streams belong to the current device.  A stream that is being captured into
// a CUDA graph is not asked for its device (that query ends the capture): the
// current device is used, so captures run with the stream's device current.
class DeviceScope {
 public:
  DeviceScope() = default;
  DeviceScope(const DeviceScope &) = delete;
  DeviceScope &operator=(const DeviceScope &) = delete;
  ~DeviceScope() {
    if (restore_ >= 0) (void)cudaSetDevice(restore_);
  }

  cudaError_t enter(cudaStream_t stream) {
    cudaError_t e = cudaGetDevice(&device_);
    if (e != cudaSuccess) return e;
    const uintptr_t s = reinterpret_cast<uintptr_t>(stream);
    if (s == 0 || s == reinterpret_cast<uintptr_t>(cudaStreamLegacy) ||
        s == reinterpret_cast<uintptr_t>(cudaStreamPerThread))
      return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return e;
    if (cs != cudaStreamCaptureStatusNone) return cudaSuccess;
    int dev = -1;
    e = cudaStreamGetDevice(stream, &dev);
    if (e != cudaSuccess) return e;
    if (dev == device_) return cudaSuccess;
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    restore_ = device_;
    device_ = dev;
    return cudaSuccess;
  }

  // The device the call's kernels are launched on.
  int device() const { return device_; }

 private:
  int device_ = -1;
  int restore_ = -1;
};

// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda)
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

CUresult encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank,
                           void *base, const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                           const cuuint32_t *box, CUtensorMapSwizzle swizzle) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return CUDA_ERROR_NOT_FOUND;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return g_encode(map, dtype, rank, base, dims, strides_bytes, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// ---------------------------------------------------------------------------
// Validation helpers
// ---------------------------------------------------------------------------
static bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

static pkv_status make_geometry(const pkv_attn_params *p, int64_t num_blocks, Geometry *g) {
  if (!p) return PKV_ERR_INVALID;
  if (p->num_heads <= 0 || p->num_kv_heads <= 0 || p->num_heads % p->num_kv_heads != 0)
    return PKV_ERR_INVALID;
  if (p->dtype != PKV_FP16 && p->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (p->head_size != 64 && p->head_size != 128) return PKV_ERR_UNSUPPORTED;
  if (p->block_size != 16 && p->block_size != 32) return PKV_ERR_UNSUPPORTED;
  if (!std::isfinite(p->scale) || p->scale <= 0.f) return PKV_ERR_INVALID;
  if (num_blocks <= 0) return PKV_ERR_INVALID;
  if (num_blocks * p->block_size > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  if (p->alibi_slopes && !aligned(p->alibi_slopes, 4)) return PKV_ERR_INVALID;
  if (p->non_causal != 0 && p->non_causal != 1) return PKV_ERR_INVALID;
  if (p->non_causal && p->sliding_window > 0) return PKV_ERR_UNSUPPORTED;
  if (p->kv_cache_dtype != PKV_CACHE_AUTO && p->kv_cache_dtype != PKV_CACHE_FP8_E4M3)
    return PKV_ERR_UNSUPPORTED;
  const bool fp8 = p->kv_cache_dtype == PKV_CACHE_FP8_E4M3;
  if (fp8 && (!std::isfinite(p->k_scale) || !std::isfinite(p->v_scale) || p->k_scale <= 0.f ||
              p->v_scale <= 0.f))
    return PKV_ERR_INVALID;
  g->H = p->num_heads;
  g->KVH = p->num_kv_heads;
  g->QPK = p->num_heads / p->num_kv_heads;
  g->D = p->head_size;
  g->BS = p->block_size;
  g->dtype = p->dtype;
  g->scale = p->scale;
  g->alibi = p->alibi_slopes;
  g->window = p->sliding_window > 0 ? p->sliding_window : 0;
  g->non_causal = p->non_causal;
  g->num_blocks = num_blocks;
  g->row_elems = static_cast<int64_t>(g->KVH) * g->D;
  g->block_elems = g->row_elems * g->BS;
  g->fp8 = fp8;
  g->k_scale = fp8 ? p->k_scale : 1.f;
  g->v_scale = fp8 ? p->v_scale : 1.f;
  g->elem_bytes = fp8 ? 1 : 2;
  g->row_bytes = g->row_elems * g->elem_bytes;
  g->block_bytes = g->block_elems * g->elem_bytes;
  return PKV_OK;
}

static pkv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

constexpr int32_t kMaxMultiQueryLen = 64;  // tokens per sequence of a multi-token decode

}  // namespace pkv

using namespace pkv;

extern "C" {

int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

const char *pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_BOUNDS: return "device-side index out of range";
    case PKV_ERR_TIMEOUT: return "device-side bounded wait timed out";
  }
  return "unknown status";
}

pkv_status kv_cache_write(const void *key, const void *value, int64_t num_tokens, void *kv_cache,
                          int64_t num_blocks, const int64_t *slot_mapping,
                          const pkv_attn_params *params, pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, num_blocks, &g);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_INVALID;
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !kv_cache || !slot_mapping) return PKV_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PKV_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  cudaError_t e = scope.enter(s);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return from_cuda(launch_kv_write(key, value, num_tokens, kv_cache, slot_mapping, g, s));
}

size_t paged_attn_decode_workspace_size(int32_t num_seqs, int32_t max_seq_len,
                                        const pkv_attn_params *params) {
  Geometry g;
  if (make_geometry(params, 1, &g) != PKV_OK || num_seqs <= 0 || max_seq_len < 0) return 0;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) dev.sms = 152;
  return plan_decode(num_seqs, 1, max_seq_len, g, dev.sms).workspace_bytes;
}

pkv_status paged_attn_decode(void *out, const void *query, int32_t num_seqs, const void *kv_cache,
                             int64_t num_blocks, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *seq_lens,
                             int32_t max_seq_len, const pkv_attn_params *params, void *workspace,
                             size_t workspace_bytes, pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, num_blocks, &g);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || max_seq_len < 0 || max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !query || !kv_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID;
  if (!aligned(out, 16) || !aligned(query, 16) || !aligned(kv_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return PKV_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  cudaError_t e = scope.enter(s);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  DeviceInfo dev;
  e = current_device_info(&dev);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  const DecodePlan plan = plan_decode(num_seqs, 1, max_seq_len, g, dev.sms);
  if (plan.workspace_bytes > 0 &&
      (!workspace || workspace_bytes < plan.workspace_bytes || !aligned(workspace, 16)))
    return PKV_ERR_INVALID;
  return from_cuda(launch_decode(out, query, num_seqs, 1, kv_cache, block_tables,
                                 max_blocks_per_seq, seq_lens, g, plan, workspace, s));
}

pkv_status paged_attn_decode_noalloc(void *out, const void *query, int32_t num_seqs,
                                     const void *kv_cache, int64_t num_blocks,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const int32_t *seq_lens, int32_t max_seq_len,
                                     const pkv_attn_params *params, pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, num_blocks, &g);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || max_seq_len < 0 || max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID;
  if (num_seqs == 0) return PKV_OK;
  // The scratch array of the device the kernels will run on: the stream's
  // device, current for the rest of this call (a capturing stream: the
  // current device, which the capture must run on).
  DeviceScope scope;
  cudaError_t e = scope.enter(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  if (paged_attn_decode_workspace_size(num_seqs, max_seq_len, params) >
      PKV_DECODE_STATIC_SCRATCH_BYTES)
    return PKV_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  size_t scratch_bytes = 0;
  if (static_decode_scratch(scope.device(), &scratch, &scratch_bytes) != cudaSuccess)
    return PKV_ERR_CUDA;
  return paged_attn_decode(out, query, num_seqs, kv_cache, num_blocks, block_tables,
                           max_blocks_per_seq, seq_lens, max_seq_len, params, scratch,
                           scratch_bytes, stream);
}

static bool multi_args_supported(const Geometry &g, int32_t query_len) {
  return !g.non_causal && query_len >= 1 && query_len <= kMaxMultiQueryLen;
}

size_t paged_attn_decode_multi_workspace_size(int32_t num_seqs, int32_t query_len,
                                              int32_t max_seq_len,
                                              const pkv_attn_params *params) {
  Geometry g;
  if (make_geometry(params, 1, &g) != PKV_OK || num_seqs <= 0 || max_seq_len < 0 ||
      !multi_args_supported(g, query_len))
    return 0;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) dev.sms = 152;
  return plan_decode(num_seqs, query_len, max_seq_len, g, dev.sms).workspace_bytes;
}

pkv_status paged_attn_decode_multi(void *out, const void *query, int32_t num_seqs,
                                   int32_t query_len, const void *kv_cache, int64_t num_blocks,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *seq_lens, int32_t max_seq_len,
                                   const pkv_attn_params *params, void *workspace,
                                   size_t workspace_bytes, pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, num_blocks, &g);
  if (st != PKV_OK) return st;
  if (query_len < 1 || num_seqs < 0 || num_seqs > 65535 || max_seq_len < 0 ||
      max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID;
  if (!multi_args_supported(g, query_len)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (static_cast<int64_t>(num_seqs) * query_len > 0x7fffffffLL / g.H) return PKV_ERR_UNSUPPORTED;
  if (!out || !query || !kv_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID;
  if (!aligned(out, 16) || !aligned(query, 16) || !aligned(kv_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return PKV_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  cudaError_t e = scope.enter(s);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  DeviceInfo dev;
  e = current_device_info(&dev);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  const DecodePlan plan = plan_decode(num_seqs, query_len, max_seq_len, g, dev.sms);
  if (plan.workspace_bytes > 0 &&
      (!workspace || workspace_bytes < plan.workspace_bytes || !aligned(workspace, 16)))
    return PKV_ERR_INVALID;
  return from_cuda(launch_decode(out, query, num_seqs, query_len, kv_cache, block_tables,
                                 max_blocks_per_seq, seq_lens, g, plan, workspace, s));
}

constexpr int32_t kMaxDcpWorld = 1024;

size_t paged_attn_decode_dcp_workspace_size(int32_t num_seqs, int32_t query_len,
                                            int32_t max_seq_len, int32_t dcp_world_size,
                                            const pkv_attn_params *params) {
  Geometry g;
  if (make_geometry(params, 1, &g) != PKV_OK || num_seqs <= 0 || max_seq_len < 0 ||
      !multi_args_supported(g, query_len) || dcp_world_size < 1 || dcp_world_size > kMaxDcpWorld)
    return 0;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) dev.sms = 152;
  return plan_decode(num_seqs, query_len, max_seq_len, g, dev.sms, dcp_world_size)
      .workspace_bytes;
}

pkv_status paged_attn_decode_dcp_partial(float *part_o, float *part_ml, const void *query,
                                         int32_t num_seqs, int32_t query_len,
                                         const void *kv_cache, int64_t num_blocks,
                                         const int32_t *block_tables,
                                         int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                         int32_t max_seq_len, int32_t dcp_world_size,
                                         int32_t dcp_rank, const pkv_attn_params *params,
                                         void *workspace, size_t workspace_bytes,
                                         pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, num_blocks, &g);
  if (st != PKV_OK) return st;
  if (query_len < 1 || num_seqs < 0 || num_seqs > 65535 || max_seq_len < 0 ||
      max_blocks_per_seq <= 0 || dcp_world_size < 1 || dcp_world_size > kMaxDcpWorld ||
      dcp_rank < 0 || dcp_rank >= dcp_world_size)
    return PKV_ERR_INVALID;
  if (!multi_args_supported(g, query_len)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (static_cast<int64_t>(num_seqs) * query_len > 0x7fffffffLL / g.H) return PKV_ERR_UNSUPPORTED;
  if (!part_o || !part_ml || !query || !kv_cache || !block_tables || !seq_lens)
    return PKV_ERR_INVALID;
  if (!aligned(part_o, 16) || !aligned(part_ml, 8) || !aligned(query, 16) ||
      !aligned(kv_cache, 16) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return PKV_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  cudaError_t e = scope.enter(s);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  DeviceInfo dev;
  e = current_device_info(&dev);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  const DecodePlan plan =
      plan_decode(num_seqs, query_len, max_seq_len, g, dev.sms, dcp_world_size);
  if (plan.workspace_bytes > 0 &&
      (!workspace || workspace_bytes < plan.workspace_bytes || !aligned(workspace, 16)))
    return PKV_ERR_INVALID;
  DcpShare share;
  share.world = dcp_world_size;
  share.rank = dcp_rank;
  share.res_o = part_o;
  share.res_ml = part_ml;
  return from_cuda(launch_decode(nullptr, query, num_seqs, query_len, kv_cache, block_tables,
                                 max_blocks_per_seq, seq_lens, g, plan, workspace, s, share));
}

pkv_status paged_attn_dcp_combine(void *out, const float *part_o, const float *part_ml,
                                  int32_t num_parts, int64_t num_rows,
                                  const pkv_attn_params *params, pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, 1, &g);
  if (st != PKV_OK) return st;
  if (num_parts < 1 || num_parts > kMaxDcpWorld || num_rows < 0) return PKV_ERR_INVALID;
  if (num_rows == 0) return PKV_OK;
  if (num_rows > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  if (!out || !part_o || !part_ml) return PKV_ERR_INVALID;
  if (!aligned(out, 16) || !aligned(part_o, 16) || !aligned(part_ml, 8)) return PKV_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  cudaError_t e = scope.enter(s);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return from_cuda(launch_dcp_combine(out, part_o, part_ml, num_parts, num_rows, g, s));
}

pkv_status paged_attn_prefill_varlen(void *out, const void *query, int64_t num_query_tokens,
                                     int32_t num_seqs,
                                     const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                     int32_t max_query_len, int32_t max_seq_len,
                                     const void *kv_cache, int64_t num_blocks,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const pkv_attn_params *params, pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, num_blocks, &g);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || max_query_len < 0 || max_seq_len < 0 ||
      max_blocks_per_seq <= 0 || num_query_tokens < 0 || num_query_tokens > 0x7fffffffLL)
    return PKV_ERR_INVALID;
  if (num_seqs == 0 || max_query_len == 0 || num_query_tokens == 0) return PKV_OK;
  if (static_cast<int64_t>(max_query_len) > 65535LL * 64) return PKV_ERR_UNSUPPORTED;
  if (!out || !query || !kv_cache || !block_tables || !cu_seqlens_q || !cu_seqlens_k)
    return PKV_ERR_INVALID;
  if (!aligned(out, 16) || !aligned(query, 16) || !aligned(kv_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return PKV_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  cudaError_t e = scope.enter(s);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return from_cuda(launch_prefill(out, query, num_query_tokens, num_seqs, cu_seqlens_q,
                                  cu_seqlens_k, max_query_len, max_seq_len, kv_cache,
                                  block_tables, max_blocks_per_seq, g, s));
}

pkv_status kv_copy_blocks(void *const *kv_caches, int32_t num_layers, int64_t num_blocks,
                          const int64_t *pairs, int64_t num_pairs, const pkv_attn_params *params,
                          pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, num_blocks, &g);
  if (st != PKV_OK) return st;
  if (num_pairs < 0 || num_layers < 0 || num_layers > 256) return PKV_ERR_INVALID;
  if (num_pairs == 0 || num_layers == 0) return PKV_OK;
  if (!kv_caches || !pairs || !aligned(pairs, 8)) return PKV_ERR_INVALID;
  for (int l = 0; l < num_layers; ++l)
    if (!kv_caches[l] || !aligned(kv_caches[l], 16)) return PKV_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  cudaError_t e = scope.enter(s);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  return from_cuda(launch_kv_copy(kv_caches, num_layers, pairs, num_pairs, g, s));
}

// Device-addressable view of a cache pointer, or nullptr.
static void *device_view(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return nullptr;
  switch (at.type) {
    case cudaMemoryTypeDevice:
      return at.device == cur ? at.devicePointer : nullptr;
    case cudaMemoryTypeManaged:
    case cudaMemoryTypeHost:
      return at.devicePointer;
    default:
      return nullptr;
  }
}

pkv_status kv_swap_blocks(const void *src_cache, int64_t src_num_blocks, void *dst_cache,
                          int64_t dst_num_blocks, const int64_t *pairs, int64_t num_pairs,
                          const pkv_attn_params *params, pkv_stream_t stream) {
  Geometry g;
  pkv_status st = make_geometry(params, std::max<int64_t>(src_num_blocks, 1), &g);
  if (st != PKV_OK) return st;
  if (num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 ||
      src_num_blocks > 0x7fffffffLL || dst_num_blocks > 0x7fffffffLL)
    return PKV_ERR_INVALID;
  if (num_pairs == 0) return PKV_OK;
  if (!src_cache || !dst_cache || !pairs) return PKV_ERR_INVALID;
  if (!aligned(src_cache, 16) || !aligned(dst_cache, 16)) return PKV_ERR_INVALID;
  std::vector<uint8_t> dst_used(static_cast<size_t>(dst_num_blocks), 0);
  for (int64_t k = 0; k < num_pairs; ++k) {
    const int64_t s = pairs[2 * k], d = pairs[2 * k + 1];
    if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks) return PKV_ERR_INVALID;
    if (dst_used[d]) return PKV_ERR_INVALID;
    dst_used[d] = 1;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  cudaError_t e = scope.enter(s);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  void *src_dev = device_view(src_cache);
  void *dst_dev = device_view(dst_cache);
  if (!src_dev || !dst_dev) return PKV_ERR_INVALID;
  return from_cuda(
      launch_kv_swap(src_dev, src_num_blocks, dst_dev, dst_num_blocks, pairs, num_pairs, g, s));
}

pkv_status pkv_check_wait_timeout(int64_t tag, pkv_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceScope scope;
  if (scope.enter(s) != cudaSuccess) return PKV_ERR_CUDA;
  return from_cuda(launch_wait_timeout_check(tag, s));
}

pkv_status pkv_device_error(int64_t *detail) {
  constexpr int kUnits = 3;
  unsigned long long words[kUnits] = {0, 0, 0};
  cudaError_t (*readers[kUnits])(unsigned long long *) = {
      read_device_error_kv_ops, read_device_error_decode, read_device_error_prefill};
  for (int k = 0; k < kUnits; ++k)
    if (readers[k](&words[k]) != cudaSuccess) return PKV_ERR_CUDA;
  for (int k = 0; k < kUnits; ++k) {
    if (words[k]) {
      if (detail) {
        int64_t v = static_cast<int64_t>(words[k] & ((1ull << 56) - 1));
        if (v & (1ll << 55)) v -= (1ll << 56);  // sign-extend the 56-bit field
        *detail = v;
      }
      return static_cast<pkv_status>(words[k] >> 56);
    }
  }
  if (detail) *detail = 0;
  return PKV_OK;
}

}  // extern "C"
