// Host-side interfaces between the libpkv translation units.  Arguments are
// validated by the front end (abi.cu) before any of these is called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

// Validated, derived view of pkv_attn_params.
struct Geometry {
  int H, KVH, QPK, D, BS;
  int dtype;  // pkv_dtype
  float scale;
  const float *alibi;
  int window;            // <= 0: none
  int non_causal;        // 1: every query row sees its whole sequence
  int64_t num_blocks;    // blocks per cache half
  int64_t row_elems;     // KVH * D
  int64_t block_elems;   // BS * KVH * D
  bool fp8;              // cache holds E4M3 codes (1 byte per element)
  float k_scale, v_scale;
  int64_t elem_bytes;    // of the cache: 2, or 1 for fp8
  int64_t row_bytes;     // one token row of the cache
  int64_t block_bytes;   // one block of one cache half
};

// Streams/devices: the SM count and opt-in shared memory of the current device.
struct DeviceInfo {
  int device;
  int sms;
  int max_smem_optin;
};
cudaError_t current_device_info(DeviceInfo *out);

// Driver entry point for cuTensorMapEncodeTiled, resolved once.
CUresult encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank,
                           void *base, const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                           const cuuint32_t *box, CUtensorMapSwizzle swizzle);

// kv_ops.cu
cudaError_t launch_kv_write(const void *key, const void *value, int64_t num_tokens, void *kv_cache,
                            const int64_t *slot_mapping, const Geometry &g, cudaStream_t stream);
cudaError_t launch_kv_copy(void *const *caches, int num_layers, const int64_t *pairs,
                           int64_t num_pairs, const Geometry &g, cudaStream_t stream);
cudaError_t launch_kv_swap(const void *src, int64_t src_blocks, void *dst, int64_t dst_blocks,
                           const int64_t *pairs_host, int64_t num_pairs, const Geometry &g,
                           cudaStream_t stream);
cudaError_t read_device_error_kv_ops(unsigned long long *out);
cudaError_t launch_wait_timeout_check(int64_t tag, cudaStream_t stream);

// decode.cu (single- and multi-token decode)
struct DecodePlan {
  int row_groups;   // 16-row groups of (token, head) rows per KV head
  int split_units;  // 16-key units per split
  int max_splits;   // grid extent over splits (1 = no split, no workspace)
  size_t workspace_bytes;
};
// Decode context parallelism: this rank's place in the group and, for a
// rank's share, where its (o, m, l) go instead of the output (world 1, rank
// 0 and null pointers: a plain decode).
struct DcpShare {
  int world = 1, rank = 0;
  float *res_o = nullptr, *res_ml = nullptr;
};
DecodePlan plan_decode(int num_seqs, int query_len, int max_seq_len, const Geometry &g, int sms,
                       int dcp_world = 1);
cudaError_t launch_decode(void *out, const void *query, int num_seqs, int query_len,
                          const void *kv_cache, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *seq_lens, const Geometry &g,
                          const DecodePlan &plan, void *workspace, cudaStream_t stream,
                          const DcpShare &dcp = DcpShare{});
cudaError_t launch_dcp_combine(void *out, const float *parts_o, const float *parts_ml,
                              int num_parts, int64_t num_rows, const Geometry &g,
                              cudaStream_t stream);
cudaError_t read_device_error_decode(unsigned long long *out);
// Device address and size of the static decode scratch of `device`, which
// must be the current device (looked up on the first call per device).
cudaError_t static_decode_scratch(int device, void **ptr, size_t *bytes);

// prefill.cu
cudaError_t launch_prefill(void *out, const void *query, int64_t num_q_tokens, int num_seqs,
                           const int32_t *cu_q, const int32_t *cu_k, int max_query_len,
                           int max_seq_len, const void *kv_cache, const int32_t *block_tables,
                           int max_blocks_per_seq, const Geometry &g, cudaStream_t stream);
cudaError_t read_device_error_prefill(unsigned long long *out);

}  // namespace pkv
