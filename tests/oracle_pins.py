"""Pins that tie the fp64 oracle to facts outside itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
something the source pages or the mathematics fix:

* values the pages print (the slot_mapping and cu-seqlens worked examples,
  stored under tests/golden/ with their citations);
* special cases that reduce to a library routine (torch's CPU
  ``scaled_dot_product_attention`` in fp64, the routine cpu_attn
  ``_run_sdpa_forward`` calls per sequence);
* closed forms (one key returns its V; constant V; a zero query averages the
  visible V; a zero query with ALiBi gives geometric weights; W = 1);
* invariants (block placement, GQA as duplicated K/V, causal append, the
  decode / prefill / chunked cross-path identities, the ALiBi (j-i) versus j
  equivalence the xformers.py ``_make_alibi_bias`` comment states, split-KV
  combine, copy/swap round trips).

``tests/test_oracle.py`` runs every pin; ``tests/test_oracle_mutations.py``
plants plausible mistakes in the oracle and checks that some pin fails.
"""
from __future__ import annotations

import math
import os

import torch
import torch.nn.functional as F

import oracle.paged_attention as O

F64 = torch.float64
HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


# ---------------------------------------------------------------------------
# helpers: lay contiguous per-sequence K/V into a paged cache through the
# oracle's own (separately pinned) cache write
# ---------------------------------------------------------------------------

def _params(H, KVH, D, bs, scale=None, slopes=None, window=0, causal=True):
    return O.AttnParams(num_heads=H, num_kv_heads=KVH, head_size=D,
                        block_size=bs,
                        scale=(1.0 / math.sqrt(D)) if scale is None else scale,
                        alibi_slopes=slopes, sliding_window=window, causal=causal)


def paged_from_contiguous(Ks, Vs, p, g, extra_blocks=3, dtype=torch.bfloat16):
    """Place sequences' K/V ([L_b, KVH, D] each) into a random block layout.

    Returns (kv_cache, block_tables).  Slots follow the scheduler's
    assignment block_table[pos // bs] * bs + pos % bs (the encoding whose
    decoding the slot_mapping worked example pins).
    """
    bs = p.block_size
    nblk = [(K.shape[0] + bs - 1) // bs for K in Ks]
    NB = sum(nblk) + extra_blocks
    perm = torch.randperm(NB, generator=g)
    tables = torch.zeros(len(Ks), max(1, max(nblk)), dtype=torch.int32)
    k = 0
    for b, n in enumerate(nblk):
        for lb in range(n):
            tables[b, lb] = int(perm[k])
            k += 1
    cache = torch.randn(2, NB, bs * p.row_elems, generator=g).to(dtype)
    for b, (K, V) in enumerate(zip(Ks, Vs)):
        L = K.shape[0]
        slots = torch.tensor([int(tables[b, j // bs]) * bs + j % bs
                              for j in range(L)], dtype=torch.int64)
        O.kv_cache_write(K.reshape(L, -1).to(dtype), V.reshape(L, -1).to(dtype),
                         cache, slots, p)
    return cache, tables


def _rand_seqs(g, lens, KVH, D, dtype=torch.bfloat16):
    Ks = [torch.randn(L, KVH, D, generator=g).to(dtype) for L in lens]
    Vs = [torch.randn(L, KVH, D, generator=g).to(dtype) for L in lens]
    return Ks, Vs


def _cu(lens):
    return torch.tensor([0] + list(torch.cumsum(torch.tensor(lens), 0)),
                        dtype=torch.int32)


def _prefill(Q, Ks, Vs, qlens, p, g, rows=None):
    """Oracle prefill of sequences whose subquery is the last qlens[b] rows."""
    cache, tables = paged_from_contiguous(Ks, Vs, p, g)
    lens = [K.shape[0] for K in Ks]
    return O.paged_attn_prefill_varlen(Q, _cu(qlens), _cu(lens), cache, tables,
                                       p, rows=rows)


def _sdpa(q, K, V, p, causal):
    """torch CPU fp64 SDPA with GQA by repeat_interleave; [L, H*D]."""
    qpk = p.num_heads // p.num_kv_heads
    qq = q.to(F64).permute(1, 0, 2)[None]
    kk = K.to(F64).repeat_interleave(qpk, dim=1).permute(1, 0, 2)[None]
    vv = V.to(F64).repeat_interleave(qpk, dim=1).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(qq, kk, vv, is_causal=causal, scale=p.scale)
    return o[0].permute(1, 0, 2).reshape(q.shape[0], -1)


def _sdpa_causal(q, K, V, p):
    """Library routine: torch CPU fp64 SDPA, causal, GQA by repeat_interleave.

    q: [L, H, D]; K, V: [L, KVH, D] -> [L, H*D].
    """
    qpk = p.num_heads // p.num_kv_heads
    qq = q.to(F64).permute(1, 0, 2)[None]
    kk = K.to(F64).repeat_interleave(qpk, dim=1).permute(1, 0, 2)[None]
    vv = V.to(F64).repeat_interleave(qpk, dim=1).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(qq, kk, vv, is_causal=True,
                                       scale=p.scale)
    return o[0].permute(1, 0, 2).reshape(q.shape[0], -1)


def _close(a, b, tol=1e-10, what=""):
    err = (a - b).abs().max().item()
    assert err <= tol, f"{what}: max abs diff {err:.3e} > {tol:.1e}"


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---------------------------------------------------------------------------
# pins: printed values
# ---------------------------------------------------------------------------

def pin_slot_mapping_worked_example():
    """Slots 35, 2, 17 with block size 16 -> (2,3), (0,2), (1,1)."""
    p = _params(H=2, KVH=2, D=8, bs=16)
    rows = [tuple(int(x) for x in r.split()) for r in
            _read_golden("slot_mapping_example.txt")]
    for slot, bs, blk, off in rows:
        assert O.slot_location(slot, bs) == (blk, off), (slot, bs, blk, off)
    # the write lands each key row at that (block, offset) of the K half, and
    # each value row in the V half (token-major block reading)
    g = torch.Generator().manual_seed(0)
    T = len(rows)
    key = torch.randn(T, p.row_elems, generator=g).to(torch.bfloat16)
    val = torch.randn(T, p.row_elems, generator=g).to(torch.bfloat16)
    cache = torch.zeros(2, 3, 16 * p.row_elems, dtype=torch.bfloat16)
    O.kv_cache_write(key, val, cache, torch.tensor([r[0] for r in rows]), p)
    n = p.row_elems
    for t, (_, _, blk, off) in enumerate(rows):
        assert torch.equal(cache[0, blk, off * n:(off + 1) * n].view(torch.int16),
                           key[t].view(torch.int16))
        assert torch.equal(cache[1, blk, off * n:(off + 1) * n].view(torch.int16),
                           val[t].view(torch.int16))
    written = sum(int((cache[h].view(torch.int16) != 0).any(-1).sum())
                  for h in range(2))
    assert written <= 6


def pin_negative_slot_is_skipped():
    p = _params(H=2, KVH=2, D=8, bs=4)
    cache = torch.zeros(2, 2, 4 * p.row_elems, dtype=torch.float16)
    k = torch.ones(2, p.row_elems, dtype=torch.float16)
    O.kv_cache_write(k, k, cache, torch.tensor([-1, 5]), p)
    assert int((cache != 0).sum()) == 2 * p.row_elems


def pin_cu_seqlens_worked_example():
    """Lengths [4, 6] <-> cumulative start locations [0, 4, 10]."""
    lines = _read_golden("cu_seqlens_example.txt")
    lens = [int(x) for x in lines[0].split(":")[1].split()]
    cu = [int(x) for x in lines[1].split(":")[1].split()]
    assert O.lengths_from_cu(torch.tensor(cu)) == lens


# ---------------------------------------------------------------------------
# pins: library routine (SDPA) special cases
# ---------------------------------------------------------------------------

def pin_prefill_equals_sdpa_causal():
    """c = 0 prefill, GQA 2, ragged lengths over several blocks."""
    g = torch.Generator().manual_seed(1)
    p = _params(H=4, KVH=2, D=16, bs=4, scale=0.37)
    lens = [1, 7, 13]
    Ks, Vs = _rand_seqs(g, lens, p.num_kv_heads, p.head_size)
    Q = torch.randn(sum(lens), p.num_heads * p.head_size, generator=g).to(
        torch.bfloat16)
    out = _prefill(Q, Ks, Vs, lens, p, g)
    a = 0
    for L, K, V in zip(lens, Ks, Vs):
        ref = _sdpa_causal(Q[a:a + L].view(L, p.num_heads, p.head_size), K, V, p)
        _close(out[a:a + L], ref, what=f"prefill L={L}")
        a += L


def pin_noncausal_prefill_equals_sdpa():
    """Encoder attention (cpu_attn _run_sdpa_forward with is_causal off):
    every row sees the whole sequence."""
    g = torch.Generator().manual_seed(16)
    p = _params(H=4, KVH=2, D=16, bs=4, scale=0.3, causal=False)
    lens = [1, 6, 13]
    Ks, Vs = _rand_seqs(g, lens, p.num_kv_heads, p.head_size)
    Q = torch.randn(sum(lens), p.num_heads * p.head_size, generator=g).to(torch.bfloat16)
    out = _prefill(Q, Ks, Vs, lens, p, g)
    a = 0
    for L, K, V in zip(lens, Ks, Vs):
        ref = _sdpa(Q[a:a + L].view(L, p.num_heads, p.head_size), K, V, p, causal=False)
        _close(out[a:a + L], ref, what=f"non-causal L={L}")
        a += L
    # a chunk of the last rows sees the same full sequence
    chunk = _prefill(Q[a - 4:a], [Ks[-1]], [Vs[-1]], [4], p, g)
    _close(chunk, out[a - 4:a], tol=1e-13, what="non-causal chunk")


def pin_decode_equals_sdpa_last_row():
    """Decode at length L is the last row of the causal SDPA of length L."""
    g = torch.Generator().manual_seed(2)
    p = _params(H=8, KVH=2, D=16, bs=4, scale=0.25)
    lens = [1, 5, 9, 16]
    Ks, Vs = _rand_seqs(g, lens, p.num_kv_heads, p.head_size)
    cache, tables = paged_from_contiguous(Ks, Vs, p, g)
    q = torch.randn(len(lens), p.num_heads * p.head_size, generator=g).to(
        torch.bfloat16)
    out = O.paged_attn_decode(q, cache, tables,
                              torch.tensor(lens, dtype=torch.int32), p)
    for b, (L, K, V) in enumerate(zip(lens, Ks, Vs)):
        qf = torch.randn(L, p.num_heads, p.head_size, generator=g).to(
            torch.bfloat16)
        qf[-1] = q[b].view(p.num_heads, p.head_size)
        ref = _sdpa_causal(qf, K, V, p)[-1]
        _close(out[b], ref, what=f"decode L={L}")


# ---------------------------------------------------------------------------
# pins: closed forms
# ---------------------------------------------------------------------------

def pin_single_key_returns_its_value():
    g = torch.Generator().manual_seed(3)
    p = _params(H=4, KVH=4, D=8, bs=4, slopes=[0.5, 0.25, 0.125, 1.0])
    Ks, Vs = _rand_seqs(g, [1], 4, 8)
    cache, tables = paged_from_contiguous(Ks, Vs, p, g)
    q = torch.randn(1, 32, generator=g).to(torch.bfloat16)
    out = O.paged_attn_decode(q, cache, tables, torch.tensor([1]), p)
    assert torch.equal(out[0], Vs[0][0].to(F64).reshape(-1))


def pin_constant_value_returns_it():
    g = torch.Generator().manual_seed(4)
    p = _params(H=2, KVH=1, D=8, bs=4, slopes=[0.3, 0.05], window=5)
    L = 11
    Ks, _ = _rand_seqs(g, [L], 1, 8)
    c = torch.randn(1, 1, 8, generator=g).to(torch.bfloat16)
    Vs = [c.expand(L, 1, 8).clone()]
    Q = torch.randn(L, 16, generator=g).to(torch.bfloat16)
    out = _prefill(Q, Ks, Vs, [L], p, g)
    ref = c.to(F64).reshape(1, 8).repeat(L, 2)
    _close(out, ref, tol=1e-12, what="constant V")


def pin_zero_query_averages_visible_values():
    """q = 0: uniform weights over the window_lo(i)..i keys (W = 3)."""
    g = torch.Generator().manual_seed(5)
    p = _params(H=1, KVH=1, D=8, bs=4, window=3)
    L = 10
    Ks, Vs = _rand_seqs(g, [L], 1, 8)
    Q = torch.zeros(L, 8, dtype=torch.bfloat16)
    out = _prefill(Q, Ks, Vs, [L], p, g)
    V = Vs[0].to(F64)[:, 0]
    for i in range(L):
        lo = max(0, i - 2)
        _close(out[i], V[lo:i + 1].mean(0), tol=1e-12, what=f"mean row {i}")


def pin_zero_query_alibi_geometric_weights():
    """q = 0 with ALiBi slope a: weight of key i-m is e^{-a m} / Z,
    Z = (1 - e^{-a n}) / (1 - e^{-a}) for n visible keys."""
    g = torch.Generator().manual_seed(6)
    slopes = [0.5, 0.0625]
    p = _params(H=2, KVH=1, D=8, bs=4, slopes=slopes)
    L = 9
    Ks, Vs = _rand_seqs(g, [L], 1, 8)
    q = torch.zeros(1, 16, dtype=torch.bfloat16)
    cache, tables = paged_from_contiguous(Ks, Vs, p, g)
    out = O.paged_attn_decode(q, cache, tables, torch.tensor([L]), p)
    V = Vs[0].to(F64)[:, 0]
    for h, a in enumerate(slopes):
        Z = (1 - math.exp(-a * L)) / (1 - math.exp(-a))
        ref = sum(math.exp(-a * m) * V[L - 1 - m] for m in range(L)) / Z
        _close(out[0, h * 8:(h + 1) * 8], ref, tol=1e-12, what=f"alibi h={h}")


def pin_window_one_returns_own_value():
    g = torch.Generator().manual_seed(7)
    p = _params(H=2, KVH=1, D=8, bs=4, window=1)
    L = 7
    Ks, Vs = _rand_seqs(g, [L], 1, 8)
    Q = torch.randn(L, 16, generator=g).to(torch.bfloat16)
    out = _prefill(Q, Ks, Vs, [L], p, g)
    V = Vs[0].to(F64)[:, 0]
    assert torch.equal(out, V.repeat(1, 2))


# ---------------------------------------------------------------------------
# pins: invariants
# ---------------------------------------------------------------------------

def pin_window_at_least_length_is_no_window():
    g = torch.Generator().manual_seed(8)
    L = 12
    Ks, Vs = _rand_seqs(g, [L], 2, 8)
    Q = torch.randn(L, 32, generator=g).to(torch.bfloat16)
    a = _prefill(Q, Ks, Vs, [L], _params(4, 2, 8, 4, window=L),
                 torch.Generator().manual_seed(0))
    b = _prefill(Q, Ks, Vs, [L], _params(4, 2, 8, 4, window=0),
                 torch.Generator().manual_seed(0))
    assert torch.equal(a, b)
    c = _prefill(Q, Ks, Vs, [L], _params(4, 2, 8, 4, window=L - 1),
                 torch.Generator().manual_seed(0))
    assert not torch.equal(a[-1], c[-1])


def pin_block_placement_invariance():
    g = torch.Generator().manual_seed(9)
    p = _params(H=4, KVH=2, D=8, bs=4, slopes=[0.5, 0.25, 0.1, 0.01], window=6)
    lens = [3, 10, 17]
    Ks, Vs = _rand_seqs(g, lens, 2, 8)
    q = torch.randn(3, 32, generator=g).to(torch.bfloat16)
    sl = torch.tensor(lens, dtype=torch.int32)
    outs = []
    for seed in (11, 12, 13):
        cache, tables = paged_from_contiguous(Ks, Vs, p,
                                              torch.Generator().manual_seed(seed))
        outs.append(O.paged_attn_decode(q, cache, tables, sl, p))
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def pin_gqa_equals_duplicated_kv():
    """GQA equals MHA on K/V repeated per query head (cpu_attn
    repeat_interleave along the head axis)."""
    g = torch.Generator().manual_seed(10)
    H, KVH, D = 6, 2, 8
    lens = [5, 9]
    Ks, Vs = _rand_seqs(g, lens, KVH, D)
    Q = torch.randn(sum(lens), H * D, generator=g).to(torch.bfloat16)
    a = _prefill(Q, Ks, Vs, lens, _params(H, KVH, D, 4),
                 torch.Generator().manual_seed(1))
    Kd = [K.repeat_interleave(H // KVH, dim=1) for K in Ks]
    Vd = [V.repeat_interleave(H // KVH, dim=1) for V in Vs]
    b = _prefill(Q, Kd, Vd, lens, _params(H, H, D, 4),
                 torch.Generator().manual_seed(1))
    _close(a, b, tol=0.0, what="gqa vs duplicated")


def pin_causal_append_keeps_earlier_rows():
    g = torch.Generator().manual_seed(11)
    p = _params(H=2, KVH=1, D=8, bs=4, slopes=[0.2, 0.7])
    L1, L2 = 6, 11
    Ks, Vs = _rand_seqs(g, [L2], 1, 8)
    Q = torch.randn(L2, 16, generator=g).to(torch.bfloat16)
    short = _prefill(Q[:L1], [Ks[0][:L1]], [Vs[0][:L1]], [L1], p, g)
    long = _prefill(Q, Ks, Vs, [L2], p, g)
    _close(long[:L1], short, tol=1e-13, what="causal append")


def pin_cross_path_identities():
    """decode(L) == last row of prefill(L) == chunked (c = L-1, q = 1);
    chunked (c, q) rows == full-prefill rows c..c+q-1."""
    g = torch.Generator().manual_seed(12)
    p = _params(H=4, KVH=2, D=8, bs=4, slopes=[0.3, 0.2, 0.1, 0.05], window=7)
    L, c = 14, 9
    Ks, Vs = _rand_seqs(g, [L], 2, 8)
    Q = torch.randn(L, 32, generator=g).to(torch.bfloat16)
    full = _prefill(Q, Ks, Vs, [L], p, g)
    chunk = _prefill(Q[c:], Ks, Vs, [L - c], p, g)
    _close(chunk, full[c:], tol=1e-13, what="chunked vs full")
    last = _prefill(Q[L - 1:], Ks, Vs, [1], p, g)
    _close(last[0], full[L - 1], tol=1e-13, what="chunk of one vs full")
    cache, tables = paged_from_contiguous(Ks, Vs, p, g)
    dec = O.paged_attn_decode(Q[L - 1:], cache, tables, torch.tensor([L]), p)
    _close(dec[0], full[L - 1], tol=1e-13, what="decode vs full")


def pin_alibi_offset_equivalence():
    """slope*(j - i) and slope*j differ by a per-row constant: same output."""
    g = torch.Generator().manual_seed(13)
    D, L = 8, 9
    K = torch.randn(L, D, generator=g, dtype=F64)
    V = torch.randn(L, D, generator=g, dtype=F64)
    q = torch.randn(3, D, generator=g, dtype=F64)
    pos = [2, 5, 8]
    a = O.attend_rows(q, pos, K, V, 0.3, 0.4, 0)
    b = torch.stack([
        torch.softmax(0.3 * (K[:i + 1] @ q[r]) + 0.4 * torch.arange(i + 1, dtype=F64), 0)
        @ V[:i + 1] for r, i in enumerate(pos)])
    _close(a, b, tol=1e-13, what="alibi j-i vs j")


def pin_split_combine_equals_direct():
    g = torch.Generator().manual_seed(14)
    D, L = 8, 37
    K = torch.randn(L, D, generator=g, dtype=F64)
    V = torch.randn(L, D, generator=g, dtype=F64)
    q = torch.randn(D, generator=g, dtype=F64)
    for slope, window in ((None, 0), (0.2, 0), (None, 20), (0.05, 11)):
        ref = O.attend_rows(q[None], [L - 1], K, V, 0.5, slope, window)[0]
        for split in (1, 4, 16, 64):
            parts = O.decode_split_partials(q, K, V, L - 1, 0.5, slope, window,
                                            split)
            _close(O.combine_split_partials(parts), ref, tol=1e-12,
                   what=f"split {split}")


def pin_copy_and_swap_round_trip():
    g = torch.Generator().manual_seed(15)
    caches = [torch.randn(2, 10, 24, generator=g).to(torch.bfloat16)
              for _ in range(3)]
    before = [c.clone() for c in caches]
    pairs = [(1, 5), (1, 6), (3, 7)]
    O.kv_copy_blocks(caches, pairs)
    for c, c0 in zip(caches, before):
        for s, d in pairs:
            assert torch.equal(c[:, d].view(torch.int16), c0[:, s].view(torch.int16))
        untouched = [k for k in range(10) if k not in (5, 6, 7)]
        assert torch.equal(c[:, untouched], c0[:, untouched])
    dev = caches[0].clone()
    host = torch.zeros(2, 4, 24, dtype=torch.bfloat16)
    out_pairs = [(2, 0), (8, 1), (4, 3)]
    O.kv_swap_blocks(dev, host, out_pairs)
    assert torch.equal(host[:, 2], torch.zeros(2, 24, dtype=torch.bfloat16))
    back = torch.zeros_like(dev)
    O.kv_swap_blocks(host, back, [(d, s) for s, d in out_pairs])
    for s, _ in out_pairs:
        assert torch.equal(back[:, s].view(torch.int16), dev[:, s].view(torch.int16))


# ---------------------------------------------------------------------------
# pins: the fp8 (E4M3) cache codes
# ---------------------------------------------------------------------------

def pin_e4m3_decode_matches_library():
    """Every code's value against torch's float8_e4m3fn widening."""
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(F64)
    mine = torch.tensor([O.e4m3_decode(c) for c in range(256)], dtype=F64)
    nan = torch.isnan(lib)
    assert torch.equal(torch.isnan(mine), nan)
    assert torch.equal(mine[~nan], lib[~nan])


def pin_e4m3_encode_matches_library_in_range():
    """Nearest-even rounding against torch's float8_e4m3fn narrowing, on every
    code value, every midpoint between neighbours (the ties) and a sweep, all
    inside +-464 (torch returns NaN beyond; saturation is pinned below)."""
    vals = sorted({O.e4m3_decode(c) for c in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    pts = torch.tensor(vals + mids + [464.0], dtype=torch.float32)
    pts = torch.cat([pts, -pts, torch.linspace(-464, 464, 20001)])
    lib = pts.to(torch.float8_e4m3fn).view(torch.uint8)
    mine = torch.tensor([O.e4m3_encode(float(v)) for v in pts.tolist()], dtype=torch.uint8)
    assert torch.equal(mine, lib)


def pin_e4m3_saturation_and_specials():
    assert O.e4m3_encode(1000.0) == 0x7E and O.e4m3_encode(-1e6) == 0xFE   # +-448
    assert O.e4m3_encode(float("nan")) == 0x7F
    assert O.e4m3_encode(-0.0) == 0x80 and O.e4m3_encode(2.0 ** -10) == 0x00
    assert O.e4m3_decode(0x7E) == 448.0 and O.e4m3_decode(0x01) == 2.0 ** -9


def pin_fp8_cache_equals_bf16_cache_of_its_values():
    """Attention over an fp8 cache (code * scale) equals attention over a bf16
    cache holding the same, exactly representable, values."""
    g = torch.Generator().manual_seed(17)
    H, KVH, D, bs = 4, 2, 16, 4
    p8 = O.AttnParams(H, KVH, D, bs, 0.25, [0.5, 0.25, 0.1, 0.02], 0, True,
                      "fp8_e4m3", 0.125, 0.5)
    pb = O.AttnParams(H, KVH, D, bs, 0.25, [0.5, 0.25, 0.1, 0.02])
    L = 11
    tables = torch.tensor([[2, 0, 5]], dtype=torch.int32)
    slots = torch.tensor([int(tables[0, j // bs]) * bs + j % bs for j in range(L)])
    key = torch.randn(L, KVH * D, generator=g).to(torch.bfloat16)
    val = torch.randn(L, KVH * D, generator=g).to(torch.bfloat16)
    c8 = torch.zeros(2, 6, bs * KVH * D, dtype=torch.uint8)
    O.kv_cache_write(key, val, c8, slots, p8)
    # the bf16 cache holds code * scale, computed from the codes' bit fields
    cb = torch.zeros(2, 6, bs * KVH * D, dtype=torch.bfloat16)
    for half, sc in ((0, 0.125), (1, 0.5)):
        vals = torch.tensor([O.e4m3_decode(int(c)) * sc for c in c8[half].reshape(-1)])
        cb[half] = vals.view(6, -1).to(torch.bfloat16)
    q = torch.randn(1, H * D, generator=g).to(torch.bfloat16)
    sl = torch.tensor([L], dtype=torch.int32)
    a = O.paged_attn_decode(q, c8, tables, sl, p8)
    b = O.paged_attn_decode(q, cb, tables, sl, pb)
    _close(a, b, tol=1e-13, what="fp8 vs bf16 cache")
    # and the codes are the nearest codes of key / k_scale
    assert int(c8[0].view(6, bs, KVH * D)[2, 0, 0]) == O.e4m3_encode(float(key[0, 0]) / 0.125)


def pin_multi_decode_equals_sdpa_last_rows():
    """A decode of q tokens at length L is the last q rows of the causal SDPA
    of length L (library routine), for q = 1 .. 4."""
    g = torch.Generator().manual_seed(31)
    p = _params(H=8, KVH=2, D=16, bs=4, scale=0.3)
    lens = [4, 7, 13, 16]
    Ks, Vs = _rand_seqs(g, lens, p.num_kv_heads, p.head_size)
    cache, tables = paged_from_contiguous(Ks, Vs, p, g)
    sl = torch.tensor(lens, dtype=torch.int32)
    for q in (1, 2, 4):
        Q = torch.randn(len(lens) * q, p.num_heads * p.head_size, generator=g).to(torch.bfloat16)
        out = O.paged_attn_decode_multi(Q, cache, tables, sl, q, p)
        for b, (L, K, V) in enumerate(zip(lens, Ks, Vs)):
            qf = torch.randn(L, p.num_heads, p.head_size, generator=g).to(torch.bfloat16)
            qf[L - q:] = Q[b * q:(b + 1) * q].view(q, p.num_heads, p.head_size)
            ref = _sdpa_causal(qf, K, V, p)[L - q:]
            _close(out[b * q:(b + 1) * q], ref, what=f"multi decode q={q} L={L}")


def pin_multi_decode_cross_paths():
    """q = 1 is the single-token decode; q tokens are the chunked prefill of
    the last q rows (window and ALiBi on); padding sequences are zero."""
    g = torch.Generator().manual_seed(32)
    p = _params(H=4, KVH=2, D=8, bs=4, slopes=[0.3, 0.2, 0.1, 0.05], window=6)
    lens = [3, 9, 14]
    Ks, Vs = _rand_seqs(g, lens, 2, 8)
    cache, tables = paged_from_contiguous(Ks, Vs, p, g)
    sl = torch.tensor(lens, dtype=torch.int32)
    Q1 = torch.randn(3, 32, generator=g).to(torch.bfloat16)
    _close(O.paged_attn_decode_multi(Q1, cache, tables, sl, 1, p),
           O.paged_attn_decode(Q1, cache, tables, sl, p), tol=1e-13, what="q=1 vs decode")
    q = 3
    Q3 = torch.randn(3 * q, 32, generator=g).to(torch.bfloat16)
    pre = O.paged_attn_prefill_varlen(Q3, _cu([q] * 3), _cu(lens), cache, tables, p)
    _close(O.paged_attn_decode_multi(Q3, cache, tables, sl, q, p), pre, tol=1e-13,
           what="multi decode vs chunked prefill")
    z = O.paged_attn_decode_multi(Q3, cache, tables, torch.tensor([0, 9, 14]), q, p)
    assert torch.equal(z[:q], torch.zeros(q, 32, dtype=F64))


def pin_dcp_local_lengths_count_the_rank_tokens():
    """dcp_local_seq_len is the count of positions j < L with j % R == r,
    and the local positions enumerate exactly those (brute force)."""
    for R in (1, 2, 3, 4):
        for L in range(0, 23):
            total = 0
            for r in range(R):
                n = O.dcp_local_seq_len(L, R, r)
                assert n == sum(1 for j in range(L) if j % R == r), (L, R, r)
                assert [O.dcp_global_position(k, R, r) for k in range(n)] == \
                    [j for j in range(L) if j % R == r]
                total += n
            assert total == L


def pin_dcp_partials_combine_to_the_decode():
    """Every rank's (o, m, l) over its own keys, merged by a3, gives the
    decode over the whole sequence: single and multi-token, with window and
    ALiBi, 2 and 3 ranks; one rank alone is the plain decode."""
    from paged_kv_cache_246_gb300.workloads import shard_for_dcp
    g = torch.Generator().manual_seed(41)
    for R, q, window, slopes in ((1, 1, 0, None), (2, 1, 0, None), (3, 2, 6, [0.3, 0.1]),
                                 (2, 3, 0, [0.25, 0.05])):
        p = _params(H=2, KVH=1, D=8, bs=4, scale=0.4, slopes=slopes, window=window)
        lens = [q, 5, 13, 16]
        Ks, Vs = _rand_seqs(g, lens, 1, 8)
        cache, tables = paged_from_contiguous(Ks, Vs, p, g)
        sl = torch.tensor(lens, dtype=torch.int32)
        Q = torch.randn(len(lens) * q, 16, generator=g).to(torch.bfloat16)
        ref = O.paged_attn_decode_multi(Q, cache, tables, sl, q, p)
        parts = []
        for r, (lc, lt) in enumerate(shard_for_dcp(cache, tables, sl, 4, R)):
            parts.append(O.paged_attn_decode_dcp_partials(Q, lc, lt, sl, q, R, r, p))
        got = O.combine_dcp_partials(parts, 2, 8)
        _close(got, ref, tol=1e-12, what=f"dcp R={R} q={q}")
        if R == 1:
            _close(parts[0][0], ref, tol=1e-12, what="one rank")


def pin_empty_decode_row_is_zero():
    p = _params(H=2, KVH=1, D=4, bs=4)
    cache = torch.randn(2, 2, 16).to(torch.bfloat16)
    out = O.paged_attn_decode(torch.randn(2, 8).to(torch.bfloat16), cache,
                              torch.tensor([[0], [1]], dtype=torch.int32),
                              torch.tensor([0, 3]), p)
    assert torch.equal(out[0], torch.zeros(8, dtype=F64))
    assert torch.isfinite(out[1]).all()


ALL_PINS = {name: fn for name, fn in sorted(globals().items())
            if name.startswith("pin_") and callable(fn)}
