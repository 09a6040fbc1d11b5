"""The C ABI on the host: the library loads, exports every declared symbol,
and rejects bad arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_246_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from paged_kv_cache_246_gb300 import build_lib
        build_lib.build()
    return B.lib()


def test_header_lists_the_calls():
    names = declared_functions()
    for must in ("kv_cache_write", "paged_attn_decode", "paged_attn_prefill_varlen",
                 "kv_copy_blocks", "kv_swap_blocks", "paged_attn_decode_workspace_size"):
        assert must in names
    assert set(names) == set(B.EXPORTS)


def test_static_scratch_limit_matches_the_header():
    m = re.search(r"#define PKV_DECODE_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)",
                  open(HEADER).read())
    assert m and int(m.group(1)) << int(m.group(2)) == B.PKV_DECODE_STATIC_SCRATCH_BYTES


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.pkv_abi_version() == 3
    assert ctypes.sizeof(B.AttnParams) == 56
    for s in range(6):
        assert B.status_string(s)
    assert B.status_string(99) == "unknown status"


def _p(**kw):
    base = dict(num_heads=32, num_kv_heads=8, head_size=128, block_size=16, dtype=B.PKV_BF16,
                scale=0.088, alibi_slopes=None, sliding_window=0, non_causal=0,
                kv_cache_dtype=B.PKV_CACHE_AUTO, k_scale=1.0, v_scale=1.0)
    base.update(kw)
    return B.AttnParams(**base)


def test_params_validation(lib):
    nul = ctypes.c_void_p(0)
    write = lambda p, n=1, nb=4: lib.kv_cache_write(nul, nul, n, nul, nb, nul,
                                                    ctypes.byref(p) if p else None, nul)
    assert write(None) == B.PKV_ERR_INVALID
    assert write(_p(num_heads=6, num_kv_heads=4)) == B.PKV_ERR_INVALID
    assert write(_p(head_size=96)) == B.PKV_ERR_UNSUPPORTED
    assert write(_p(block_size=24)) == B.PKV_ERR_UNSUPPORTED
    assert write(_p(dtype=7)) == B.PKV_ERR_UNSUPPORTED
    assert write(_p(scale=float("nan"))) == B.PKV_ERR_INVALID
    assert write(_p(scale=0.0)) == B.PKV_ERR_INVALID
    assert write(_p(non_causal=1, sliding_window=8)) == B.PKV_ERR_UNSUPPORTED
    assert write(_p(non_causal=2)) == B.PKV_ERR_INVALID
    assert write(_p(kv_cache_dtype=2)) == B.PKV_ERR_UNSUPPORTED
    fp8 = dict(kv_cache_dtype=B.PKV_CACHE_FP8_E4M3)
    assert write(_p(k_scale=0.0, **fp8)) == B.PKV_ERR_INVALID
    assert write(_p(v_scale=-1.0, **fp8)) == B.PKV_ERR_INVALID
    assert write(_p(k_scale=float("inf"), **fp8)) == B.PKV_ERR_INVALID
    assert write(_p(k_scale=0.0), n=0) == B.PKV_OK   # scales unused by an "auto" cache
    assert write(_p(**fp8), n=0) == B.PKV_OK
    assert write(_p(), nb=0) == B.PKV_ERR_INVALID
    assert write(_p(), n=-1) == B.PKV_ERR_INVALID
    assert write(_p(), n=1) == B.PKV_ERR_INVALID      # null pointers
    assert write(_p(), n=0) == B.PKV_OK               # empty: nothing enqueued


def test_decode_and_prefill_validation(lib):
    nul = ctypes.c_void_p(0)
    p = _p()
    assert lib.paged_attn_decode(nul, nul, 0, nul, 4, nul, 1, nul, 0, ctypes.byref(p), nul, 0,
                                 nul) == B.PKV_OK
    assert lib.paged_attn_decode(nul, nul, 2, nul, 4, nul, 1, nul, 8, ctypes.byref(p), nul, 0,
                                 nul) == B.PKV_ERR_INVALID
    assert lib.paged_attn_decode(nul, nul, 70000, nul, 4, nul, 1, nul, 8, ctypes.byref(p), nul,
                                 0, nul) == B.PKV_ERR_INVALID
    p3 = _p(num_heads=24, num_kv_heads=8)  # any group size: here the null pointers fail
    assert lib.paged_attn_decode(nul, nul, 2, nul, 4, nul, 1, nul, 8, ctypes.byref(p3), nul, 0,
                                 nul) == B.PKV_ERR_INVALID
    assert lib.paged_attn_prefill_varlen(nul, nul, 10, 3, nul, nul, 0, 5, nul, 4, nul, 1,
                                         ctypes.byref(p), nul) == B.PKV_OK
    assert lib.paged_attn_prefill_varlen(nul, nul, 10, 3, nul, nul, 5, 5, nul, 4, nul, 1,
                                         ctypes.byref(p), nul) == B.PKV_ERR_INVALID
    assert lib.paged_attn_prefill_varlen(nul, nul, -1, 3, nul, nul, 5, 5, nul, 4, nul, 1,
                                         ctypes.byref(p), nul) == B.PKV_ERR_INVALID
    p8 = _p(kv_cache_dtype=B.PKV_CACHE_FP8_E4M3, k_scale=0.02, v_scale=0.02)
    assert lib.paged_attn_prefill_varlen(nul, nul, 10, 3, nul, nul, 0, 5, nul, 4, nul, 1,
                                         ctypes.byref(p8), nul) == B.PKV_OK
    assert lib.paged_attn_prefill_varlen(nul, nul, 10, 3, nul, nul, 5, 5, nul, 4, nul, 1,
                                         ctypes.byref(p8), nul) == B.PKV_ERR_INVALID


def test_multi_decode_validation(lib):
    nul = ctypes.c_void_p(0)
    p = _p()
    call = lambda pp, B=2, q=4: lib.paged_attn_decode_multi(nul, nul, B, q, nul, 4, nul, 1, nul,
                                                          8, ctypes.byref(pp), nul, 0, nul)
    assert call(p, B=0) == B.PKV_OK                     # empty: nothing enqueued
    assert call(p, q=0) == B.PKV_ERR_INVALID
    assert call(p, q=65) == B.PKV_ERR_UNSUPPORTED
    assert call(p) == B.PKV_ERR_INVALID                 # null pointers
    assert call(_p(non_causal=1)) == B.PKV_ERR_UNSUPPORTED
    fp8 = _p(kv_cache_dtype=B.PKV_CACHE_FP8_E4M3, k_scale=0.1, v_scale=0.1)
    assert call(fp8) == B.PKV_ERR_INVALID               # supported: null pointers
    assert call(_p(num_heads=24, num_kv_heads=8)) == B.PKV_ERR_INVALID   # any group size
    assert B.paged_attn_decode_multi_workspace_size(4, 4, 64, p) == 0   # one split
    n = B.paged_attn_decode_multi_workspace_size(128, 4, 16384, p)
    assert n > 0 and n % 256 == 0
    assert B.paged_attn_decode_multi_workspace_size(128, 0, 4096, p) == 0


def test_workspace_size_is_host_only(lib):
    p = _p()
    assert B.paged_attn_decode_workspace_size(0, 100, p) == 0
    assert B.paged_attn_decode_workspace_size(4, 64, p) == 0            # one split
    n = B.paged_attn_decode_workspace_size(256, 16384, p)
    assert n > 0 and n % 256 == 0


def test_copy_and_swap_validation(lib):
    nul = ctypes.c_void_p(0)
    p = _p()
    assert lib.kv_copy_blocks(None, 1, 8, nul, 0, ctypes.byref(p), nul) == B.PKV_OK
    assert lib.kv_copy_blocks(None, 300, 8, nul, 1, ctypes.byref(p), nul) == B.PKV_ERR_INVALID
    pairs = (ctypes.c_int64 * 4)(0, 1, 2, 1)  # destination 1 twice
    fake = ctypes.c_void_p(1 << 20)
    assert lib.kv_swap_blocks(fake, 8, fake, 8, pairs, 2, ctypes.byref(p),
                              nul) == B.PKV_ERR_INVALID
    pairs = (ctypes.c_int64 * 2)(9, 0)        # source out of range
    assert lib.kv_swap_blocks(fake, 8, fake, 8, pairs, 1, ctypes.byref(p),
                              nul) == B.PKV_ERR_INVALID


def test_split_plan_at_the_bench_shapes(lib):
    """The split planner (host only; 152 SMs without a device): splits of up
    to 4096 keys, halved while the grid would hold fewer than 8 CTAs per SM.
    The workspace is rows x splits x (head_size + 2) fp32 values, each part
    rounded up to 256 bytes."""
    p, win = _p(), _p(sliding_window=4096)
    # 2048 (sequence, KV head) items fill the GPU with one split each
    assert B.paged_attn_decode_workspace_size(256, 4096, p) == 0
    assert B.paged_attn_decode_multi_workspace_size(128, 4, 4096, p) == 0
    # 512 items: 4096-key splits are halved to 2048; 257 units (a window
    # start can straddle one) make three splits
    three = 64 * 32 * 3
    assert B.paged_attn_decode_workspace_size(64, 4096, p) == three * 128 * 4 + three * 2 * 4
    assert B.paged_attn_decode_workspace_size(64, 32768, win) == three * 128 * 4 + three * 2 * 4
    # 32 items over 65536 keys: halved down to 1024-key splits, 65 of them
    many = 4 * 32 * 65
    assert B.paged_attn_decode_workspace_size(4, 65536, p) == many * 128 * 4 + many * 2 * 4
