"""GPU parity: every call of the C ABI against the fp64 oracle on the same
seeded inputs.  Cache writes and block moves must be bit-exact; attention
outputs within max-abs 2e-2 and mean-abs 2e-3 (fp32 accumulation, outputs
rounded to fp16/bf16).  Sizes span several tiles / splits and ragged tails."""
import math

import pytest
import torch

import oracle as O
from paged_kv_cache_246_gb300 import binding as B
from paged_kv_cache_246_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_helpers import (DEV, CudaRun, assert_close, assert_no_device_error,  # noqa: E402
                             oracle_cache_after_write, oracle_params)


def small(seed, *, dtype=torch.bfloat16, H=8, KVH=2, D=128, bs=16, seq_lens, query_lens=None,
          P=0, alibi=False, window=0, num_blocks=None, causal=True, multi=0):
    g = torch.Generator().manual_seed(seed)
    if query_lens is None:
        query_lens = [multi or 1] * len(seq_lens)
    return W.build(name=f"case{seed}", g=g, dtype=dtype, num_heads=H, num_kv_heads=KVH,
                   head_size=D, block_size=bs, seq_lens=seq_lens, query_lens=query_lens,
                   num_prefill_seqs=P, alibi=alibi, sliding_window=window, num_blocks=num_blocks,
                   causal=causal, multi_query_len=multi)


def rand_lens(seed, n, lo, hi):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# ---------------------------------------------------------------------------
# a1: cache write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_kv_cache_write_bit_exact(cfg):
    w = W.make_config(cfg, scale_down=1 if cfg == 1 else 16)
    r = CudaRun(w)
    r.write()
    assert_no_device_error("write")
    ref = oracle_cache_after_write(w)
    assert torch.equal(r.cache.cpu().view(torch.int16), ref.view(torch.int16))


def test_kv_cache_write_padding_slots_and_empty():
    w = small(11, seq_lens=[5, 9, 33], query_lens=[5, 9, 33], P=3)
    w.slot_mapping[::3] = -1  # padding tokens
    r = CudaRun(w)
    r.write()
    B.kv_cache_write(r.key[:0], r.value[:0], r.cache, r.slots[:0], r.p)  # empty: no-op
    assert_no_device_error("write padding")
    ref = oracle_cache_after_write(w)
    assert torch.equal(r.cache.cpu().view(torch.int16), ref.view(torch.int16))


def test_kv_cache_write_repeatable():
    w = W.make_config(2, scale_down=32)
    outs = []
    for _ in range(3):
        r = CudaRun(w)
        r.write()
        outs.append(r.cache.cpu())
    assert all(torch.equal(outs[0].view(torch.int16), o.view(torch.int16)) for o in outs[1:])


# ---------------------------------------------------------------------------
# a2 + a3: decode
# ---------------------------------------------------------------------------

DECODE_CASES = {
    "tiny_fp16_cfg1": lambda: W.make_config(1),
    "qpk4_multi_split": lambda: small(21, H=32, KVH=8, seq_lens=rand_lens(1, 12, 1, 600)),
    "qpk1": lambda: small(22, H=4, KVH=4, seq_lens=rand_lens(2, 7, 1, 300)),
    "qpk2_d64": lambda: small(23, H=4, KVH=2, D=64, seq_lens=rand_lens(3, 9, 1, 400)),
    "qpk8_groups": lambda: small(24, H=16, KVH=2, seq_lens=rand_lens(4, 5, 1, 700)),
    "fp16_d128": lambda: small(25, dtype=torch.float16, seq_lens=rand_lens(5, 6, 1, 500)),
    "block32": lambda: small(26, bs=32, seq_lens=rand_lens(6, 6, 1, 900)),
    "alibi": lambda: small(27, H=8, KVH=2, alibi=True, seq_lens=rand_lens(7, 6, 1, 800)),
    "window": lambda: small(28, window=100, seq_lens=rand_lens(8, 8, 1, 900)),
    "window_alibi_bs32": lambda: small(29, bs=32, window=77, alibi=True,
                                       seq_lens=rand_lens(9, 8, 1, 700)),
    "one_token_seqs": lambda: small(30, seq_lens=[1, 1, 2, 17]),
    "long_single": lambda: small(31, H=32, KVH=8, seq_lens=[5000]),
    "climbing_scores": lambda: climbing(small(33, H=32, KVH=8, seq_lens=[40, 700, 2100])),
    "window_ge_len": lambda: small(32, window=4096, seq_lens=rand_lens(10, 4, 1, 300)),
    "qpk3": lambda: small(35, H=24, KVH=8, seq_lens=rand_lens(12, 6, 1, 700)),
    "qpk6_fp16_d64": lambda: small(36, dtype=torch.float16, H=12, KVH=2, D=64,
                                   seq_lens=rand_lens(13, 6, 1, 500)),
    "qpk32_two_row_groups": lambda: small(37, H=32, KVH=1, seq_lens=rand_lens(14, 4, 1, 900)),
}


@pytest.mark.parametrize("case", sorted(DECODE_CASES))
def test_decode_parity(case):
    w = DECODE_CASES[case]()
    r = CudaRun(w)
    r.write()
    out = r.decode()
    assert_no_device_error(case)
    ref_cache = oracle_cache_after_write(w)
    q, bt, sl, _ = w.decode_slices()
    ref = O.paged_attn_decode(q, ref_cache, bt, sl, oracle_params(w))
    assert_close(out, ref, case)


def test_decode_zero_length_rows_are_zero():
    w = small(33, seq_lens=[3, 40, 2])
    r = CudaRun(w)
    r.write()
    P = 0
    sl = w.seq_lens.clone()
    sl[1] = 0
    out = torch.full_like(r.query, float("nan"))
    n = B.paged_attn_decode_workspace_size(3, 40, r.p)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
    B.paged_attn_decode(out, r.query, r.cache, r.tables, sl.to(DEV), 40, r.p, ws)
    assert_no_device_error("zero rows")
    assert torch.equal(out[1].cpu(), torch.zeros_like(out[1].cpu()))
    ref = O.paged_attn_decode(w.query, oracle_cache_after_write(w), w.block_tables, sl,
                              oracle_params(w))
    assert_close(out, ref, "zero rows")


def test_decode_split_invariance():
    """A loose max_seq_len changes the split plan, not the result."""
    w = small(34, H=32, KVH=8, seq_lens=rand_lens(11, 10, 200, 2000))
    r = CudaRun(w)
    r.write()
    a = r.decode()
    b = r.decode(max_seq_len=8 * int(w.seq_lens.max()))
    assert_no_device_error("split invariance")
    err = (a.double() - b.double()).abs().max().item()
    assert err <= 2e-2


# ---------------------------------------------------------------------------
# f3: multi-token (speculative) decode
# ---------------------------------------------------------------------------

def mlens(seed, n, q, hi):
    return [max(q, x) for x in rand_lens(seed, n, 1, hi)]


MULTI_CASES = {
    "q2_qpk4": lambda: small(121, H=32, KVH=8, multi=2, seq_lens=mlens(1, 9, 2, 600)),
    "q4_qpk4_multi_split": lambda: small(122, H=32, KVH=8, multi=4, seq_lens=mlens(2, 6, 4, 3000)),
    "q1_is_decode": lambda: small(123, H=32, KVH=8, multi=1, seq_lens=mlens(3, 7, 1, 700)),
    "q3_qpk1": lambda: small(124, H=4, KVH=4, multi=3, seq_lens=mlens(4, 7, 3, 400)),
    "q5_qpk4_two_row_groups": lambda: small(125, H=8, KVH=2, multi=5, seq_lens=mlens(5, 5, 5, 900)),
    "q4_qpk8_d64": lambda: small(126, H=16, KVH=2, D=64, multi=4, seq_lens=mlens(6, 5, 4, 700)),
    "q3_qpk6_odd_group": lambda: small(127, H=12, KVH=2, multi=3, seq_lens=mlens(7, 4, 3, 500)),
    "fp16_bs32": lambda: small(128, dtype=torch.float16, bs=32, multi=4,
                               seq_lens=mlens(8, 6, 4, 900)),
    "window_alibi": lambda: small(129, window=100, alibi=True, multi=4,
                                  seq_lens=mlens(9, 8, 4, 900)),
    "window_bs32_q6": lambda: small(130, bs=32, window=37, multi=6, seq_lens=mlens(10, 6, 6, 800)),
    "exact_lengths": lambda: small(131, multi=4, seq_lens=[4, 5, 16, 17, 31, 33]),
    "long_single": lambda: small(132, H=32, KVH=8, multi=4, seq_lens=[5000]),
    "q16_qpk4": lambda: small(133, H=32, KVH=8, multi=16, seq_lens=mlens(11, 3, 16, 600)),
}


@pytest.mark.parametrize("case", sorted(MULTI_CASES))
def test_decode_multi_parity(case):
    w = MULTI_CASES[case]()
    r = CudaRun(w)
    r.write()
    out = r.decode_multi()
    assert_no_device_error(case)
    ref_cache = oracle_cache_after_write(w)
    ref = O.paged_attn_decode_multi(w.query, ref_cache, w.block_tables, w.seq_lens,
                                    w.multi_query_len, oracle_params(w))
    assert_close(out, ref, case)


FP8_MULTI_CASES = {
    "q4_qpk4": lambda: fp8(small(141, H=32, KVH=8, multi=4, seq_lens=mlens(21, 8, 4, 2500))),
    "q1_qpk4": lambda: fp8(small(142, H=32, KVH=8, multi=1, seq_lens=mlens(22, 8, 1, 900))),
    "q3_qpk8_d64_fp16": lambda: fp8(small(143, dtype=torch.float16, H=16, KVH=2, D=64, multi=3,
                                          seq_lens=mlens(23, 5, 3, 700))),
    "window_alibi_bs32": lambda: fp8(small(144, bs=32, window=90, alibi=True, multi=4,
                                           seq_lens=mlens(24, 6, 4, 900))),
    "huge_queries": lambda: scaled_q(fp8(small(145, multi=2, seq_lens=mlens(25, 4, 2, 300))),
                                     3e4),
    "tiny_queries": lambda: scaled_q(fp8(small(146, multi=2, seq_lens=mlens(26, 4, 2, 300))),
                                     1e-6),
}


@pytest.mark.parametrize("case", sorted(FP8_MULTI_CASES))
def test_decode_multi_fp8_parity(case):
    w = FP8_MULTI_CASES[case]()
    r = CudaRun(w)
    r.write()
    out = r.decode_multi()
    assert_no_device_error(case)
    ref_cache = oracle_cache_after_write(w)
    ref = O.paged_attn_decode_multi(w.query, ref_cache, w.block_tables, w.seq_lens,
                                    w.multi_query_len, oracle_params(w))
    assert_close(out, ref, case)


def test_decode_multi_q1_matches_decode_and_split_invariance():
    w = small(134, H=32, KVH=8, multi=1, seq_lens=mlens(12, 10, 1, 2000))
    r = CudaRun(w)
    r.write()
    a = r.decode_multi()
    b = r.decode()
    c = r.decode_multi(max_seq_len=8 * int(w.seq_lens.max()))  # other split plan
    assert_no_device_error("multi q=1")
    assert (a.double() - b.double()).abs().max().item() <= 2e-2
    assert (a.double() - c.double()).abs().max().item() <= 2e-2


def test_decode_multi_padding_and_short_lengths():
    w = small(135, multi=4, seq_lens=[40, 9, 70])
    r = CudaRun(w)
    r.write()
    sl = w.seq_lens.clone()
    sl[1] = 0                      # padding sequence: zero rows
    out = torch.full_like(r.query, float("nan"))
    B.paged_attn_decode_multi(out, r.query, r.cache, r.tables, sl.to(DEV), 4, 70, r.p)
    assert_no_device_error("multi padding")
    assert torch.equal(out[4:8].cpu(), torch.zeros_like(out[4:8].cpu()))
    ref = O.paged_attn_decode_multi(w.query, oracle_cache_after_write(w), w.block_tables, sl, 4,
                                    oracle_params(w))
    assert_close(out, ref, "multi padding")
    sl[1] = 3                      # shorter than its 4 query tokens: reported, zero rows
    B.paged_attn_decode_multi(out, r.query, r.cache, r.tables, sl.to(DEV), 4, 70, r.p)
    torch.cuda.synchronize()
    st, detail = B.device_error()
    assert st == B.PKV_ERR_BOUNDS and detail == 1
    assert torch.equal(out[4:8].cpu(), torch.zeros_like(out[4:8].cpu()))


# ---------------------------------------------------------------------------
# a4: varlen / chunked prefill
# ---------------------------------------------------------------------------

def chunked(seed, ctx, q, **kw):
    return small(seed, seq_lens=[c + n for c, n in zip(ctx, q)], query_lens=q, P=len(q), **kw)


def climbing(w, q_gain=2.0, per_pos=1 / 40):
    """Scores that climb with the key position: every cached context key row
    scaled by 1 + j * per_pos (j its position), queries by q_gain.  The
    running max then grows by far more than 2^8 in p from key tile to key
    tile, which drives the kernels' rescaling (and, in prefill, the pass that
    redoes a tile whose exponents were taken against a stale max)."""
    bs = w.block_size
    row = w.kv_cache.shape[2] // bs
    ctx = (w.seq_lens - w.query_lens).tolist()
    for b, c in enumerate(ctx):
        for j in range(c):
            blk, off = int(w.block_tables[b, j // bs]), j % bs
            seg = w.kv_cache[0, blk, off * row:(off + 1) * row]
            seg.copy_((seg.float() * (1 + j * per_pos)).to(seg.dtype))
    w.query = (w.query.float() * q_gain).to(w.query.dtype)
    return w


def falling(w, q_gain=2.0, per_pos=1 / 40):
    """Scores that fall with the key position: every cached context key row
    scaled by 1 + (c - 1 - j) * per_pos (c the context length), queries by
    q_gain, so the farthest keys score highest.  With ALiBi the kernel visits
    the nearest key tile first; these rows then pass the reference max on
    later (farther) tiles, which drives the max-first pass and the rescale in
    that order."""
    bs = w.block_size
    row = w.kv_cache.shape[2] // bs
    ctx = (w.seq_lens - w.query_lens).tolist()
    for b, c in enumerate(ctx):
        for j in range(c):
            blk, off = int(w.block_tables[b, j // bs]), j % bs
            seg = w.kv_cache[0, blk, off * row:(off + 1) * row]
            seg.copy_((seg.float() * (1 + (c - 1 - j) * per_pos)).to(seg.dtype))
    w.query = (w.query.float() * q_gain).to(w.query.dtype)
    return w


PREFILL_CASES = {
    "varlen_qpk4": lambda: small(41, H=32, KVH=8, seq_lens=[1, 17, 64, 65, 130, 300],
                                 query_lens=[1, 17, 64, 65, 130, 300], P=6),
    "chunked_ctx": lambda: chunked(42, [0, 5, 64, 100, 333], [70, 1, 64, 129, 40]),
    "chunked_alibi": lambda: chunked(43, [13, 200, 0], [150, 64, 90], alibi=True, H=8, KVH=2),
    "window": lambda: small(44, window=50, seq_lens=[300, 77], query_lens=[300, 77], P=2),
    "window_chunked_alibi": lambda: chunked(45, [120, 9], [200, 33], window=64, alibi=True),
    "fp16_d64": lambda: chunked(46, [0, 31], [100, 70], dtype=torch.float16, D=64, H=4, KVH=2),
    "block32_qpk1": lambda: chunked(47, [40, 0], [90, 200], bs=32, H=4, KVH=4),
    "qpk8": lambda: chunked(48, [10, 300], [257, 3], H=16, KVH=2),
    "single_row_chunks": lambda: chunked(49, [0, 10, 99, 500], [1, 1, 1, 1]),
    "climbing_scores": lambda: climbing(chunked(53, [0, 300, 700], [200, 129, 64])),
    "climbing_scores_fp16_qpk8": lambda: climbing(chunked(54, [450, 30], [100, 250],
                                                          dtype=torch.float16, H=16, KVH=2)),
    "alibi_falling_scores": lambda: falling(chunked(55, [600, 1500, 40], [130, 64, 257],
                                                    alibi=True, H=8, KVH=2)),
    "alibi_climbing_scores": lambda: climbing(chunked(57, [300, 900], [200, 70], alibi=True,
                                                      H=8, KVH=2)),
    "alibi_qpk4_long_context": lambda: chunked(56, [1000, 2500], [300, 129], alibi=True, H=32,
                                               KVH=8),
    "noncausal_varlen": lambda: small(51, H=32, KVH=8, causal=False, seq_lens=[1, 17, 129, 300],
                                      query_lens=[1, 17, 129, 300], P=4),
    "noncausal_chunked_alibi": lambda: chunked(52, [0, 70, 200], [150, 33, 257], causal=False,
                                               alibi=True),
    "noncausal_rowpair_fp16_d64": lambda: chunked(53, [5, 0], [300, 140], causal=False,
                                                  dtype=torch.float16, D=64, H=3, KVH=3),
}


@pytest.mark.parametrize("case", sorted(PREFILL_CASES))
def test_prefill_parity(case):
    w = PREFILL_CASES[case]()
    r = CudaRun(w)
    r.write()
    out = r.prefill()
    assert_no_device_error(case)
    ref_cache = oracle_cache_after_write(w)
    q, cuq, cuk, bt, _, _ = w.prefill_slices()
    ref = O.paged_attn_prefill_varlen(q, cuq, cuk, ref_cache, bt, oracle_params(w))
    assert_close(out, ref, case)


def test_prefill_last_row_equals_decode():
    """Cross-path: the last prefill row of a sequence equals its decode."""
    lens = [33, 130, 257]
    w = small(50, H=32, KVH=8, seq_lens=lens, query_lens=lens, P=3)
    r = CudaRun(w)
    r.write()
    pre = r.prefill()
    last = torch.tensor([sum(lens[:k + 1]) - 1 for k in range(3)])
    q = r.query[last.to(DEV)].contiguous()
    out = torch.empty_like(q)
    n = B.paged_attn_decode_workspace_size(3, max(lens), r.p)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
    B.paged_attn_decode(out, q, r.cache, r.tables, w.seq_lens.to(DEV), max(lens), r.p, ws)
    assert_no_device_error("cross path")
    err = (pre[last.to(DEV)].double() - out.double()).abs().max().item()
    assert err <= 2e-2


# ---------------------------------------------------------------------------
# a5, a6: block moves
# ---------------------------------------------------------------------------

def test_copy_blocks_bit_exact_all_layers():
    g = torch.Generator().manual_seed(60)
    w = small(60, seq_lens=[64, 100], num_blocks=40)
    layers = [w.kv_cache.clone() for _ in range(3)]
    for L in layers:
        L.view(-1).copy_(torch.randn(L.numel(), generator=g).to(L.dtype))
    pairs = torch.tensor([[3, 20], [3, 21], [7, 30], [0, 39], [12, 22]], dtype=torch.int64)
    dev_layers = [L.to(DEV) for L in layers]
    r = CudaRun(w)
    B.kv_copy_blocks(dev_layers, pairs.to(DEV), r.p)
    assert_no_device_error("copy")
    O.kv_copy_blocks(layers, pairs.tolist())
    for got, ref in zip(dev_layers, layers):
        assert torch.equal(got.cpu().view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("fp8", [False, True])
def test_copy_blocks_many_pairs_ragged_pieces(fp8):
    """Blocks of 24 KiB (bs 32 x 3 KV heads x 128 dims x 2 B; 12 KiB of codes
    over an fp8 cache) cut into a full and a partial piece, 700 pairs over 2
    layers (several ring turns per CTA), and one bad pair in the middle:
    recorded, skipped, every other pair copied bit-exactly."""
    g = torch.Generator().manual_seed(63)
    w = small(63, H=6, KVH=3, bs=32, seq_lens=[40], num_blocks=1500)
    dt = torch.uint8 if fp8 else w.dtype
    layers = []
    for _ in range(2):
        L = torch.empty(w.kv_cache.shape, dtype=dt)
        if fp8:
            L.copy_(torch.randint(0, 256, L.shape, generator=g, dtype=torch.uint8))
        else:
            L.view(-1).copy_(torch.randn(L.numel(), generator=g).to(L.dtype))
        layers.append(L)
    perm = torch.randperm(1500, generator=g)
    pairs = torch.stack([perm[:700], perm[700:1400]], 1).to(torch.int64)
    bad = 333
    pairs[bad, 0] = 1500 + 9                      # source beyond the pool
    dev_layers = [L.to(DEV) for L in layers]
    r = CudaRun(w)
    p = B.make_params(6, 3, 128, 32, w.dtype, w.scale, kv_cache_dtype="fp8_e4m3", k_scale=0.02,
                      v_scale=0.02) if fp8 else r.p
    B.kv_copy_blocks(dev_layers, pairs.to(DEV), p)
    torch.cuda.synchronize()
    st, detail = B.device_error()
    assert st == B.PKV_ERR_BOUNDS and detail == bad
    good = torch.cat([pairs[:bad], pairs[bad + 1:]]).tolist()
    O.kv_copy_blocks(layers, good)
    for got, ref in zip(dev_layers, layers):
        assert torch.equal(got.cpu().view(torch.uint8), ref.view(torch.uint8))


def test_swap_round_trip_pinned_host():
    w = small(61, seq_lens=[300, 200], num_blocks=64)
    r = CudaRun(w)
    host = torch.zeros((2, 16, w.kv_cache.shape[2]), dtype=w.dtype).pin_memory()
    out_pairs = torch.tensor([[5, 0], [17, 3], [40, 15], [63, 7]], dtype=torch.int64)
    B.kv_swap_blocks(r.cache, host, out_pairs, r.p)
    torch.cuda.synchronize()
    ref_host = torch.zeros_like(host)
    O.kv_swap_blocks(w.kv_cache, ref_host, out_pairs.tolist())
    assert torch.equal(host.view(torch.int16), ref_host.view(torch.int16))
    back = torch.zeros_like(r.cache)
    in_pairs = out_pairs[:, [1, 0]].contiguous()
    B.kv_swap_blocks(host, back, in_pairs, r.p)
    assert_no_device_error("swap")
    for s in out_pairs[:, 0].tolist():
        assert torch.equal(back[:, s].cpu().view(torch.int16), w.kv_cache[:, s].view(torch.int16))


def test_swap_rejects_pageable_host():
    w = small(62, seq_lens=[20], num_blocks=4)
    r = CudaRun(w)
    pageable = torch.zeros((2, 4, w.kv_cache.shape[2]), dtype=w.dtype)
    with pytest.raises(ValueError):
        B.kv_swap_blocks(r.cache, pageable, torch.tensor([[0, 0]]), r.p)


# ---------------------------------------------------------------------------
# In-kernel range checks: bad indices are recorded, never dereferenced
# ---------------------------------------------------------------------------

def test_bad_slot_is_reported_not_written():
    w = small(70, seq_lens=[8], query_lens=[8], P=1, num_blocks=2)
    r = CudaRun(w)
    before = r.cache.clone()
    bad = r.slots.clone()
    bad[3] = 2 * 16 + 5  # beyond num_blocks * block_size
    B.kv_cache_write(r.key, r.value, r.cache, bad, r.p)
    torch.cuda.synchronize()
    st, detail = B.device_error()
    assert st == B.PKV_ERR_BOUNDS and detail == 3
    assert B.device_error()[0] == B.PKV_OK  # reading cleared it
    ref = before.cpu().clone()
    slots = bad.cpu().clone()
    slots[3] = -1
    O.kv_cache_write(w.key, w.value, ref, slots, oracle_params(w))
    assert torch.equal(r.cache.cpu().view(torch.int16), ref.view(torch.int16))


def test_bad_block_table_entry_is_reported():
    w = small(71, seq_lens=[40, 40])
    r = CudaRun(w)
    r.tables[1, 1] = w.num_blocks + 7
    r.decode()
    torch.cuda.synchronize()
    assert B.device_error()[0] == B.PKV_ERR_BOUNDS
    w2 = small(72, seq_lens=[40], query_lens=[40], P=1)
    r2 = CudaRun(w2)
    r2.tables[0, 2] = -5
    r2.prefill()
    torch.cuda.synchronize()
    assert B.device_error()[0] == B.PKV_ERR_BOUNDS


# ---------------------------------------------------------------------------
# fp8 (E4M3) cache: write is bit-exact, decode and block moves over codes
# ---------------------------------------------------------------------------

def fp8(w, k_scale=0.02, v_scale=0.03):
    """The same workload over an fp8 cache: codes of its context drawn as in
    workload 7, new keys/values quantised by the write."""
    g = torch.Generator().manual_seed(len(w.name) * 7919 + int(w.seq_lens.sum()))
    cache = torch.zeros(w.kv_cache.shape, dtype=torch.uint8)
    for half, sc in ((0, k_scale), (1, v_scale)):
        x = torch.randn(cache[half].numel(), generator=g) / sc
        cache[half].view(-1).copy_(x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8))
    w.kv_cache = cache
    w.kv_cache_dtype, w.k_scale, w.v_scale = "fp8_e4m3", k_scale, v_scale
    return w


FP8_WRITE_CASES = {
    "cfg7": lambda: W.make_config(7, scale_down=32),
    "prefill_bf16": lambda: fp8(small(81, seq_lens=[5, 9, 33], query_lens=[5, 9, 33], P=3)),
    "fp16_d64_bs32": lambda: fp8(small(82, dtype=torch.float16, D=64, bs=32, H=4, KVH=2,
                                       seq_lens=[40, 70], query_lens=[40, 70], P=2)),
    # scales small enough that a few percent of the quotients pass 448
    "saturating": lambda: fp8(small(83, seq_lens=[64, 17], query_lens=[64, 17], P=2),
                              k_scale=0.005, v_scale=0.004),
}


@pytest.mark.parametrize("case", sorted(FP8_WRITE_CASES))
def test_kv_cache_write_fp8_bit_exact(case):
    w = FP8_WRITE_CASES[case]()
    if case == "prefill_bf16":
        w.slot_mapping[::4] = -1
    r = CudaRun(w)
    r.write()
    assert_no_device_error(case)
    ref = oracle_cache_after_write(w)
    got = r.cache.cpu()
    assert got.dtype == torch.uint8
    assert torch.equal(got, ref), int((got != ref).sum())
    if case == "saturating":   # the case does reach the saturated codes
        assert ((ref == 0x7E) | (ref == 0xFE)).any()


FP8_DECODE_CASES = {
    "cfg7": lambda: W.make_config(7, scale_down=16),
    "qpk4_multi_split": lambda: fp8(small(91, H=32, KVH=8, seq_lens=rand_lens(21, 12, 1, 900))),
    "qpk1": lambda: fp8(small(92, H=4, KVH=4, seq_lens=rand_lens(22, 7, 1, 300))),
    "qpk2_d64": lambda: fp8(small(93, H=4, KVH=2, D=64, seq_lens=rand_lens(23, 9, 1, 600))),
    "qpk8_fp16": lambda: fp8(small(94, dtype=torch.float16, H=16, KVH=2,
                                   seq_lens=rand_lens(24, 5, 1, 700))),
    "block32_alibi": lambda: fp8(small(95, bs=32, alibi=True, seq_lens=rand_lens(25, 6, 1, 900))),
    "window": lambda: fp8(small(96, window=100, seq_lens=rand_lens(26, 8, 1, 900))),
    "long_single": lambda: fp8(small(97, H=32, KVH=8, seq_lens=[5000])),
    # four rows or fewer per KV head: the lo query terms ride in rows 4..7
    "huge_queries_qpk4": lambda: scaled_q(fp8(small(98, seq_lens=rand_lens(27, 6, 1, 700))), 3e4),
    "tiny_queries_qpk2": lambda: scaled_q(fp8(small(99, H=4, KVH=2, seq_lens=rand_lens(28, 6, 1, 700))),
                                          1e-6),
}


@pytest.mark.parametrize("case", sorted(FP8_DECODE_CASES))
def test_decode_fp8_parity(case):
    w = FP8_DECODE_CASES[case]()
    r = CudaRun(w)
    r.write()
    out = r.decode()
    assert_no_device_error(case)
    ref_cache = oracle_cache_after_write(w)
    assert torch.equal(r.cache.cpu(), ref_cache)
    q, bt, sl, _ = w.decode_slices()
    ref = O.paged_attn_decode(q, ref_cache, bt, sl, oracle_params(w))
    assert_close(out, ref, case)


def test_fp8_copy_and_swap_move_codes():
    w = fp8(small(98, seq_lens=[300, 200], num_blocks=64))
    r = CudaRun(w)
    pairs = torch.tensor([[3, 20], [7, 30], [0, 63]], dtype=torch.int64)
    B.kv_copy_blocks([r.cache], pairs.to(DEV), r.p)
    ref = w.kv_cache.clone()
    O.kv_copy_blocks([ref], pairs.tolist())
    assert torch.equal(r.cache.cpu(), ref)
    host = torch.zeros((2, 8, w.kv_cache.shape[2]), dtype=torch.uint8).pin_memory()
    out_pairs = torch.tensor([[5, 0], [40, 7]], dtype=torch.int64)
    B.kv_swap_blocks(r.cache, host, out_pairs, r.p)
    assert_no_device_error("fp8 moves")
    ref_host = torch.zeros_like(host)
    O.kv_swap_blocks(ref, ref_host, out_pairs.tolist())
    assert torch.equal(host, ref_host)


def scaled_q(w, f):
    """Queries times f, softmax scale divided by f: the same scores, query
    magnitudes far outside fp16's normal range (f = 3e4 or 1e-6)."""
    w.query = (w.query.float() * f).to(w.dtype)
    w.scale = w.scale / f
    return w


FP8_PREFILL_CASES = {
    "varlen_qpk4": lambda: fp8(small(101, H=32, KVH=8, seq_lens=[1, 17, 64, 65, 130, 300],
                                     query_lens=[1, 17, 64, 65, 130, 300], P=6)),
    "chunked_ctx": lambda: fp8(chunked(102, [0, 5, 64, 100, 333], [70, 1, 64, 129, 40])),
    "chunked_alibi": lambda: fp8(chunked(103, [13, 200, 0], [150, 64, 90], alibi=True, H=8,
                                         KVH=2)),
    "window_chunked": lambda: fp8(chunked(104, [120, 9], [200, 33], window=64)),
    "fp16_d64": lambda: fp8(chunked(105, [0, 31], [100, 70], dtype=torch.float16, D=64, H=4,
                                    KVH=2)),
    "bf16_d64_alibi": lambda: fp8(chunked(106, [40, 0], [90, 200], D=64, alibi=True)),
    "block32_qpk1": lambda: fp8(chunked(107, [40, 0], [90, 200], bs=32, H=4, KVH=4)),
    "noncausal_rowpair": lambda: fp8(chunked(108, [5, 0], [300, 140], causal=False, H=3,
                                             KVH=3)),
    "huge_queries": lambda: scaled_q(fp8(chunked(109, [0, 50], [200, 77], H=8, KVH=2)), 3e4),
    "tiny_queries": lambda: scaled_q(fp8(chunked(110, [0, 50], [200, 77], H=8, KVH=2)), 1e-6),
}


@pytest.mark.parametrize("case", sorted(FP8_PREFILL_CASES))
def test_prefill_fp8_parity(case):
    w = FP8_PREFILL_CASES[case]()
    r = CudaRun(w)
    r.write()
    out = r.prefill()
    assert_no_device_error(case)
    ref_cache = oracle_cache_after_write(w)
    assert torch.equal(r.cache.cpu(), ref_cache)
    q, cuq, cuk, bt, _, _ = w.prefill_slices()
    ref = O.paged_attn_prefill_varlen(q, cuq, cuk, ref_cache, bt, oracle_params(w))
    assert_close(out, ref, case)


def test_fp8_prefill_last_row_equals_fp8_decode():
    lens = [33, 130, 257]
    w = fp8(small(111, H=32, KVH=8, seq_lens=lens, query_lens=lens, P=3))
    r = CudaRun(w)
    r.write()
    pre = r.prefill()
    last = torch.tensor([sum(lens[:k + 1]) - 1 for k in range(3)]).to(DEV)
    q = r.query[last].contiguous()
    out = torch.empty_like(q)
    n = B.paged_attn_decode_workspace_size(3, max(lens), r.p)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
    B.paged_attn_decode(out, q, r.cache, r.tables, w.seq_lens.to(DEV), max(lens), r.p, ws)
    assert_no_device_error("fp8 cross path")
    assert (pre[last].double() - out.double()).abs().max().item() <= 2e-2


def test_fp8_dtype_mismatch_rejected():
    w = fp8(small(99, seq_lens=[40], query_lens=[40], P=1))
    r = CudaRun(w)
    wide = torch.zeros(w.kv_cache.shape, dtype=w.dtype, device=DEV)
    with pytest.raises(ValueError):   # a 2-byte cache under fp8 params
        B.kv_cache_write(r.key, r.value, wide, r.slots, r.p)
    with pytest.raises(ValueError):
        r.p.kv_cache_dtype = B.PKV_CACHE_AUTO
        B.kv_cache_write(r.key, r.value, r.cache, r.slots, r.p)


def test_a_wait_that_runs_out_reports_timeout_and_the_device_stays_usable():
    """Failure detection without a fault: a bounded wait on a barrier nothing
    completes gives up after its one-second bound and records
    PKV_ERR_TIMEOUT; work launched afterwards still matches the oracle."""
    assert B.device_error()[0] == B.PKV_OK
    B.check_wait_timeout(4242)
    torch.cuda.synchronize()
    st, detail = B.device_error()
    assert st == B.PKV_ERR_TIMEOUT and detail == 4242
    assert B.device_error()[0] == B.PKV_OK   # reading cleared it
    w = small(150, H=32, KVH=8, seq_lens=rand_lens(30, 6, 1, 700))
    r = CudaRun(w)
    r.write()
    out = r.decode()
    assert_no_device_error("after the timeout")
    q, bt, sl, _ = w.decode_slices()
    ref = O.paged_attn_decode(q, oracle_cache_after_write(w), bt, sl, oracle_params(w))
    assert_close(out, ref, "after the timeout")


# ---------------------------------------------------------------------------
# Non-finite values in unused slots (the tail of each sequence's last block)
# must not reach any output: their weights are exactly 0, and 0 * NaN = NaN
# ---------------------------------------------------------------------------

def poison_stale_slots(w, cache):
    """NaN (fp8: the NaN code 0x7F) in every slot past a sequence's end in its
    last block, in both halves of the device cache."""
    bs = w.block_size
    row = w.kv_cache.shape[2] // bs
    for b, L in enumerate(w.seq_lens.tolist()):
        if L == 0 or L % bs == 0:
            continue
        pb = int(w.block_tables[b, (L - 1) // bs])
        seg = cache[:, pb, (L % bs) * row:]
        if cache.dtype == torch.uint8:
            seg.fill_(0x7F)
        else:
            seg.fill_(float("nan"))


STALE_CASES = {
    "decode": lambda: small(160, H=32, KVH=8, seq_lens=[5, 17, 40, 301, 999]),
    "decode_fp8": lambda: fp8(small(161, H=32, KVH=8, seq_lens=[5, 17, 40, 301, 999])),
    "multi_q4": lambda: small(162, H=32, KVH=8, multi=4, seq_lens=[5, 17, 40, 301, 999]),
    "multi_q3_fp8_bs32": lambda: fp8(small(163, bs=32, multi=3, seq_lens=[4, 33, 70, 501])),
    "prefill": lambda: chunked(164, [0, 5, 100], [17, 60, 29]),
    "prefill_fp8": lambda: fp8(chunked(165, [0, 5, 100], [17, 60, 29])),
}


@pytest.mark.parametrize("case", sorted(STALE_CASES))
def test_non_finite_unused_slots_do_not_leak(case):
    w = STALE_CASES[case]()
    r = CudaRun(w)
    r.write()
    poison_stale_slots(w, r.cache)
    if case.startswith("prefill"):
        out = r.prefill()
        q, cuq, cuk, bt, _, _ = w.prefill_slices()
        ref = O.paged_attn_prefill_varlen(q, cuq, cuk, oracle_cache_after_write(w), bt,
                                          oracle_params(w))
    elif case.startswith("multi"):
        out = r.decode_multi()
        ref = O.paged_attn_decode_multi(w.query, oracle_cache_after_write(w), w.block_tables,
                                        w.seq_lens, w.multi_query_len, oracle_params(w))
    else:
        out = r.decode()
        q, bt, sl, _ = w.decode_slices()
        ref = O.paged_attn_decode(q, oracle_cache_after_write(w), bt, sl, oracle_params(w))
    assert_no_device_error(case)
    assert_close(out, ref, case)   # includes the finiteness check
