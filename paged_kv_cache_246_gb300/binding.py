"""Thin ctypes binding of libpkv.so (declared in include/pkv.h).

Argument marshalling only: each function checks the torch tensors it is given
(device, dtype, shape, contiguity), passes their data pointers, sizes and the
current CUDA stream to the C entry point of the same name, and raises
``PkvError`` on a non-OK status.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.  Loading fails loudly if the
library has not been built (``python -m paged_kv_cache_246_gb300.build_lib``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")

PKV_OK, PKV_ERR_INVALID, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_BOUNDS, PKV_ERR_TIMEOUT = range(6)
PKV_FP16, PKV_BF16 = 0, 1
PKV_CACHE_AUTO, PKV_CACHE_FP8_E4M3 = 0, 1
PKV_DECODE_STATIC_SCRATCH_BYTES = 64 << 20   # include/pkv.h: paged_attn_decode_noalloc's limit
_DTYPES = {torch.float16: PKV_FP16, torch.bfloat16: PKV_BF16}

# Every function include/pkv.h declares.
EXPORTS = ("kv_cache_write", "paged_attn_decode", "paged_attn_decode_workspace_size",
           "paged_attn_decode_noalloc", "paged_attn_decode_multi",
           "paged_attn_decode_multi_workspace_size", "paged_attn_decode_dcp_partial",
           "paged_attn_decode_dcp_workspace_size", "paged_attn_dcp_combine",
           "paged_attn_prefill_varlen", "kv_copy_blocks", "kv_swap_blocks",
           "pkv_status_string", "pkv_device_error", "pkv_abi_version",
           "pkv_check_wait_timeout")


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class AttnParams(ctypes.Structure):
    """Mirror of pkv_attn_params."""
    _fields_ = [("num_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_size", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("alibi_slopes", ctypes.c_void_p), ("sliding_window", ctypes.c_int32),
                ("non_causal", ctypes.c_int32), ("kv_cache_dtype", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once; raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "python -m paged_kv_cache_246_gb300.build_lib")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(AttnParams)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "kv_cache_write": (i32, [vp, vp, i64, vp, i64, vp, P, vp]),
            "paged_attn_decode": (i32, [vp, vp, i32, vp, i64, vp, i32, vp, i32, P, vp, sz, vp]),
            "paged_attn_decode_workspace_size": (sz, [i32, i32, P]),
            "paged_attn_decode_noalloc": (i32, [vp, vp, i32, vp, i64, vp, i32, vp, i32, P, vp]),
            "paged_attn_decode_multi": (i32, [vp, vp, i32, i32, vp, i64, vp, i32, vp, i32, P, vp,
                                              sz, vp]),
            "paged_attn_decode_multi_workspace_size": (sz, [i32, i32, i32, P]),
            "paged_attn_decode_dcp_partial": (i32, [vp, vp, vp, i32, i32, vp, i64, vp, i32, vp,
                                                    i32, i32, i32, P, vp, sz, vp]),
            "paged_attn_decode_dcp_workspace_size": (sz, [i32, i32, i32, i32, P]),
            "paged_attn_dcp_combine": (i32, [vp, vp, vp, i32, i64, P, vp]),
            "paged_attn_prefill_varlen": (i32, [vp, vp, i64, i32, vp, vp, i32, i32, vp, i64, vp,
                                                i32, P, vp]),
            "kv_copy_blocks": (i32, [vp, i32, i64, vp, i64, P, vp]),
            "kv_swap_blocks": (i32, [vp, i64, vp, i64, vp, i64, P, vp]),
            "pkv_status_string": (ctypes.c_char_p, [i32]),
            "pkv_device_error": (i32, [ctypes.POINTER(ctypes.c_int64)]),
            "pkv_abi_version": (i32, []),
            "pkv_check_wait_timeout": (i32, [i64, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype=None, ndim=None, cuda=True) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_params(num_heads: int, num_kv_heads: int, head_size: int, block_size: int,
                dtype: torch.dtype, scale: float, alibi_slopes: Optional[torch.Tensor] = None,
                sliding_window: int = 0, non_causal: bool = False,
                kv_cache_dtype: str = "auto", k_scale: float = 1.0,
                v_scale: float = 1.0) -> AttnParams:
    """pkv_attn_params; alibi_slopes is a CUDA fp32 tensor [num_heads] or None.
    kv_cache_dtype "auto" (the model dtype) or "fp8_e4m3" (uint8 cache of
    E4M3 codes with k_scale / v_scale).

    The caller keeps alibi_slopes alive while the params are in use."""
    if kv_cache_dtype not in ("auto", "fp8_e4m3"):
        raise ValueError(f"unsupported kv_cache_dtype {kv_cache_dtype}")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    ptr = None
    if alibi_slopes is not None:
        _need(alibi_slopes, "alibi_slopes", torch.float32, 1)
        if alibi_slopes.numel() != num_heads:
            raise ValueError("alibi_slopes must have num_heads entries")
        ptr = alibi_slopes.data_ptr()
    return AttnParams(num_heads, num_kv_heads, head_size, block_size, _DTYPES[dtype],
                      float(scale), ptr, int(sliding_window or 0), int(bool(non_causal)),
                      PKV_CACHE_FP8_E4M3 if kv_cache_dtype == "fp8_e4m3" else PKV_CACHE_AUTO,
                      float(k_scale), float(v_scale))


def _cache_blocks(kv_cache: torch.Tensor, p: AttnParams) -> int:
    if kv_cache.dim() != 3 or kv_cache.shape[0] != 2:
        raise ValueError("kv_cache must be [2, num_blocks, block_size*num_kv_heads*head_size]")
    if kv_cache.shape[2] != p.block_size * p.num_kv_heads * p.head_size:
        raise ValueError("kv_cache block size does not match params")
    if kv_cache.element_size() != (1 if p.kv_cache_dtype == PKV_CACHE_FP8_E4M3 else 2):
        raise ValueError("kv_cache element size does not match kv_cache_dtype")
    return int(kv_cache.shape[1])


def kv_cache_write(key: torch.Tensor, value: torch.Tensor, kv_cache: torch.Tensor,
                   slot_mapping: torch.Tensor, params: AttnParams, stream=None) -> None:
    for t, n in ((key, "key"), (value, "value"), (kv_cache, "kv_cache")):
        _need(t, n)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    nb = _cache_blocks(kv_cache, params)
    T = key.shape[0]
    row = params.num_kv_heads * params.head_size
    if key.numel() != T * row or value.numel() != T * row or slot_mapping.numel() != T:
        raise ValueError("key/value/slot_mapping sizes disagree")
    cache_dtype = torch.uint8 if params.kv_cache_dtype == PKV_CACHE_FP8_E4M3 else key.dtype
    if value.dtype != key.dtype or kv_cache.dtype != cache_dtype:
        raise ValueError("key/value dtype must match each other and the cache")
    _check(lib().kv_cache_write(key.data_ptr(), value.data_ptr(), T, kv_cache.data_ptr(), nb,
                                slot_mapping.data_ptr(), ctypes.byref(params), _stream(stream)),
           "kv_cache_write")


def paged_attn_decode_workspace_size(num_seqs: int, max_seq_len: int, params: AttnParams) -> int:
    return int(lib().paged_attn_decode_workspace_size(num_seqs, max_seq_len,
                                                      ctypes.byref(params)))


def paged_attn_decode(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                      params: AttnParams, workspace: Optional[torch.Tensor] = None,
                      stream=None) -> None:
    for t, n in ((out, "out"), (query, "query"), (kv_cache, "kv_cache")):
        _need(t, n)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    nb = _cache_blocks(kv_cache, params)
    B = seq_lens.numel()
    hd = params.num_heads * params.head_size
    if query.numel() != B * hd or out.numel() != B * hd or block_tables.shape[0] != B:
        raise ValueError("query/out/block_tables sizes disagree with seq_lens")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(lib().paged_attn_decode(out.data_ptr(), query.data_ptr(), B, kv_cache.data_ptr(), nb,
                                   block_tables.data_ptr(), int(block_tables.shape[1]),
                                   seq_lens.data_ptr(), int(max_seq_len), ctypes.byref(params),
                                   ws_ptr, ws_bytes, _stream(stream)),
           "paged_attn_decode")


def paged_attn_decode_noalloc(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor,
                              block_tables: torch.Tensor, seq_lens: torch.Tensor,
                              max_seq_len: int, params: AttnParams, stream=None) -> None:
    """paged_attn_decode without a workspace, for callers that may not
    allocate device memory: the split partials go to the library's static
    device scratch (PKV_DECODE_STATIC_SCRATCH_BYTES per GPU, shared by all
    calls; calls that overlap on the GPU race on it).  Sizes that need more
    scratch raise PkvError with PKV_ERR_UNSUPPORTED."""
    for t, n in ((out, "out"), (query, "query"), (kv_cache, "kv_cache")):
        _need(t, n)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    nb = _cache_blocks(kv_cache, params)
    B = seq_lens.numel()
    hd = params.num_heads * params.head_size
    if query.numel() != B * hd or out.numel() != B * hd or block_tables.shape[0] != B:
        raise ValueError("query/out/block_tables sizes disagree with seq_lens")
    _check(lib().paged_attn_decode_noalloc(out.data_ptr(), query.data_ptr(), B,
                                           kv_cache.data_ptr(), nb, block_tables.data_ptr(),
                                           int(block_tables.shape[1]), seq_lens.data_ptr(),
                                           int(max_seq_len), ctypes.byref(params),
                                           _stream(stream)),
           "paged_attn_decode_noalloc")


def paged_attn_decode_multi_workspace_size(num_seqs: int, query_len: int, max_seq_len: int,
                                           params: AttnParams) -> int:
    return int(lib().paged_attn_decode_multi_workspace_size(num_seqs, query_len, max_seq_len,
                                                            ctypes.byref(params)))


def paged_attn_decode_multi(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor, query_len: int,
                            max_seq_len: int, params: AttnParams,
                            workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Uniform batch of decodes of query_len tokens per sequence; query/out
    rows b * query_len + t."""
    for t, n in ((out, "out"), (query, "query"), (kv_cache, "kv_cache")):
        _need(t, n)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    nb = _cache_blocks(kv_cache, params)
    B = seq_lens.numel()
    hd = params.num_heads * params.head_size
    rows = B * int(query_len)
    if query.numel() != rows * hd or out.numel() != rows * hd or block_tables.shape[0] != B:
        raise ValueError("query/out/block_tables sizes disagree with seq_lens and query_len")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(lib().paged_attn_decode_multi(out.data_ptr(), query.data_ptr(), B, int(query_len),
                                         kv_cache.data_ptr(), nb, block_tables.data_ptr(),
                                         int(block_tables.shape[1]), seq_lens.data_ptr(),
                                         int(max_seq_len), ctypes.byref(params), ws_ptr, ws_bytes,
                                         _stream(stream)),
           "paged_attn_decode_multi")


def paged_attn_decode_dcp_workspace_size(num_seqs: int, query_len: int, max_seq_len: int,
                                         dcp_world_size: int, params: AttnParams) -> int:
    return int(lib().paged_attn_decode_dcp_workspace_size(num_seqs, query_len, max_seq_len,
                                                          dcp_world_size, ctypes.byref(params)))


def paged_attn_decode_dcp_partial(part_o: torch.Tensor, part_ml: torch.Tensor,
                                  query: torch.Tensor, kv_cache: torch.Tensor,
                                  block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                  query_len: int, max_seq_len: int, dcp_world_size: int,
                                  dcp_rank: int, params: AttnParams,
                                  workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """This rank's share (fp32 o [rows * heads, head_size], (m, l) [rows * heads, 2])
    of a decode whose sequences' tokens are spread over dcp_world_size ranks;
    seq_lens are the global lengths, kv_cache / block_tables the rank's own."""
    for t, n in ((query, "query"), (kv_cache, "kv_cache")):
        _need(t, n)
    _need(part_o, "part_o", torch.float32)
    _need(part_ml, "part_ml", torch.float32)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    nb = _cache_blocks(kv_cache, params)
    B = seq_lens.numel()
    rows = B * int(query_len)
    hd = params.num_heads * params.head_size
    if (query.numel() != rows * hd or part_o.numel() != rows * hd or
            part_ml.numel() != rows * params.num_heads * 2 or block_tables.shape[0] != B):
        raise ValueError("query/part_o/part_ml/block_tables sizes disagree")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _need(workspace, "workspace")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(lib().paged_attn_decode_dcp_partial(
        part_o.data_ptr(), part_ml.data_ptr(), query.data_ptr(), B, int(query_len),
        kv_cache.data_ptr(), nb, block_tables.data_ptr(), int(block_tables.shape[1]),
        seq_lens.data_ptr(), int(max_seq_len), int(dcp_world_size), int(dcp_rank),
        ctypes.byref(params), ws_ptr, ws_bytes, _stream(stream)), "paged_attn_decode_dcp_partial")


def paged_attn_dcp_combine(out: torch.Tensor, parts_o: torch.Tensor, parts_ml: torch.Tensor,
                           params: AttnParams, stream=None) -> None:
    """out [rows, heads * head_size] from the ranks' shares stacked rank-major:
    parts_o [P, rows * heads, head_size], parts_ml [P, rows * heads, 2]."""
    _need(out, "out")
    _need(parts_o, "parts_o", torch.float32)
    _need(parts_ml, "parts_ml", torch.float32)
    P = int(parts_o.shape[0])
    rh = params.num_heads
    rows = out.numel() // (rh * params.head_size)
    if (parts_o.numel() != P * rows * rh * params.head_size or
            parts_ml.numel() != P * rows * rh * 2):
        raise ValueError("parts_o/parts_ml sizes disagree with out")
    _check(lib().paged_attn_dcp_combine(out.data_ptr(), parts_o.data_ptr(), parts_ml.data_ptr(),
                                        P, rows, ctypes.byref(params), _stream(stream)),
           "paged_attn_dcp_combine")


def paged_attn_prefill_varlen(out: torch.Tensor, query: torch.Tensor, cu_seqlens_q: torch.Tensor,
                              cu_seqlens_k: torch.Tensor, max_query_len: int, max_seq_len: int,
                              kv_cache: torch.Tensor, block_tables: torch.Tensor,
                              params: AttnParams, stream=None) -> None:
    for t, n in ((out, "out"), (query, "query"), (kv_cache, "kv_cache")):
        _need(t, n)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    nb = _cache_blocks(kv_cache, params)
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1 or block_tables.shape[0] < B or out.shape != query.shape:
        raise ValueError("cu_seqlens/block_tables/out sizes disagree")
    rows = query.shape[0]
    if query.numel() != rows * params.num_heads * params.head_size:
        raise ValueError("query must be [num_query_tokens, num_heads * head_size]")
    _check(lib().paged_attn_prefill_varlen(out.data_ptr(), query.data_ptr(), rows, B,
                                           cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                           int(max_query_len), int(max_seq_len),
                                           kv_cache.data_ptr(), nb, block_tables.data_ptr(),
                                           int(block_tables.shape[1]), ctypes.byref(params),
                                           _stream(stream)),
           "paged_attn_prefill_varlen")


def kv_copy_blocks(kv_caches: Sequence[torch.Tensor], pairs: torch.Tensor, params: AttnParams,
                   stream=None) -> None:
    if len(kv_caches) == 0:
        return
    nb = None
    for k, c in enumerate(kv_caches):
        _need(c, f"kv_caches[{k}]")
        n = _cache_blocks(c, params)
        if nb is not None and n != nb:
            raise ValueError("all caches must have the same number of blocks")
        nb = n
    _need(pairs, "pairs", torch.int64, 2)
    arr = (ctypes.c_void_p * len(kv_caches))(*[c.data_ptr() for c in kv_caches])
    _check(lib().kv_copy_blocks(arr, len(kv_caches), nb, pairs.data_ptr(), int(pairs.shape[0]),
                                ctypes.byref(params), _stream(stream)),
           "kv_copy_blocks")


def kv_swap_blocks(src_cache: torch.Tensor, dst_cache: torch.Tensor, pairs: torch.Tensor,
                   params: AttnParams, stream=None) -> None:
    """pairs: CPU int64 [n, 2]; src/dst: CUDA tensors or pinned CPU tensors."""
    for t, n in ((src_cache, "src_cache"), (dst_cache, "dst_cache")):
        _need(t, n, cuda=False)
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{n} must be a CUDA tensor or pinned host memory")
    _need(pairs, "pairs", torch.int64, 2, cuda=False)
    if pairs.is_cuda:
        raise ValueError("swap pairs are read on the host: pass a CPU tensor")
    sb, db = _cache_blocks(src_cache, params), _cache_blocks(dst_cache, params)
    _check(lib().kv_swap_blocks(src_cache.data_ptr(), sb, dst_cache.data_ptr(), db,
                                pairs.data_ptr(), int(pairs.shape[0]), ctypes.byref(params),
                                _stream(stream)),
           "kv_swap_blocks")


def check_wait_timeout(tag: int, stream=None) -> None:
    """Launch the bounded wait that nothing completes (pkv_check_wait_timeout)."""
    _check(lib().pkv_check_wait_timeout(int(tag), _stream(stream)), "pkv_check_wait_timeout")


def device_error() -> tuple[int, int]:
    """(status, detail) of the sticky device error word; reading clears it."""
    d = ctypes.c_int64(0)
    st = lib().pkv_device_error(ctypes.byref(d))
    return int(st), int(d.value)


def check_device_error(where: str = "device") -> None:
    st, d = device_error()
    if st != PKV_OK:
        raise PkvError(st, f"{where} (first bad index {d})")
