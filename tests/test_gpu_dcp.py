"""Decode context parallelism on one GPU: the ranks' shares computed by
paged_attn_decode_dcp_partial over per-rank caches (token j of a sequence on
rank j % R), stacked as the all-gather stacks them, merged by
paged_attn_dcp_combine: the result must match the oracle's decode over the
whole, unsharded sequences.  (The exchange itself runs between processes;
tests/test_dcp_multirank.py covers it with gloo ranks on CPU.)"""
import pytest
import torch

import oracle as O
from paged_kv_cache_246_gb300 import binding as B
from paged_kv_cache_246_gb300 import dcp as DCP
from paged_kv_cache_246_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_helpers import (DEV, CudaRun, assert_close, assert_no_device_error,  # noqa: E402
                             oracle_cache_after_write, oracle_params)


def batch(seed, *, world, q=1, H=8, KVH=2, D=128, bs=16, lens, alibi=False, window=0,
          dtype=torch.bfloat16, fp8=False):
    g = torch.Generator().manual_seed(seed)
    extra = dict(kv_cache_dtype="fp8_e4m3", k_scale=0.02, v_scale=0.02) if fp8 else {}
    w = W.build(name=f"dcp{seed}", g=g, dtype=dtype, num_heads=H, num_kv_heads=KVH, head_size=D,
                block_size=bs, seq_lens=lens, query_lens=[q] * len(lens), num_prefill_seqs=0,
                alibi=alibi, sliding_window=window, multi_query_len=q, **extra)
    return w, world


def lens_of(seed, n, q, hi):
    g = torch.Generator().manual_seed(seed)
    return [max(q, int(x)) for x in torch.randint(1, hi + 1, (n,), generator=g)]


CASES = {
    "r1_is_plain_decode": lambda: batch(201, world=1, H=32, KVH=8, lens=lens_of(1, 6, 1, 900)),
    "r2_qpk4": lambda: batch(202, world=2, H=32, KVH=8, lens=lens_of(2, 8, 1, 3000)),
    "r3_q4_window_alibi": lambda: batch(203, world=3, q=4, alibi=True, window=200,
                                        lens=lens_of(3, 6, 4, 1500)),
    "r4_short_sequences": lambda: batch(204, world=4, lens=[1, 2, 3, 5, 17]),
    "r2_fp8": lambda: batch(205, world=2, H=32, KVH=8, fp8=True, lens=lens_of(5, 6, 1, 2000)),
    "r2_fp16_d64_bs32": lambda: batch(206, world=2, dtype=torch.float16, D=64, bs=32, q=2,
                                      lens=lens_of(6, 5, 2, 1200)),
}


def poison_past_local_ends(shards, seq_lens, bs, R):
    """Copies of the per-rank caches with NaN (fp8: the NaN code 0x7F) in
    every slot past a rank's last token in its last local block."""
    out = []
    for r, (lc, lt) in enumerate(shards):
        lc = lc.clone()
        row = lc.shape[2] // bs
        for b, L in enumerate(seq_lens.tolist()):
            Lr = max(0, (L - r + R - 1) // R)
            if Lr == 0 or Lr % bs == 0:
                continue
            seg = lc[:, int(lt[b, (Lr - 1) // bs]), (Lr % bs) * row:]
            if lc.dtype == torch.uint8:
                seg.fill_(0x7F)
            else:
                seg.fill_(float("nan"))
        out.append((lc, lt))
    return out


@pytest.mark.parametrize("case", sorted(CASES))
def test_dcp_shares_merge_to_the_decode(case):
    _check_dcp(case, poison=False)


@pytest.mark.parametrize("case", ["r2_fp8", "r2_qpk4", "r3_q4_window_alibi"])
def test_dcp_non_finite_unused_slots_do_not_leak(case):
    _check_dcp(case, poison=True)


def _check_dcp(case, poison):
    w, R = CASES[case]()
    if w.kv_cache_dtype == "fp8_e4m3":   # context codes as the fp8 workloads draw them
        g = torch.Generator().manual_seed(9)
        for half in (0, 1):
            x = torch.randn(w.kv_cache[half].numel(), generator=g) / 0.02
            w.kv_cache[half].view(-1).copy_(
                x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8))
    q = w.multi_query_len
    r = CudaRun(w)
    r.write()                                   # the new tokens, into the whole cache
    assert_no_device_error(case + " write")
    whole = r.cache.cpu()
    shards = W.shard_for_dcp(whole, w.block_tables, w.seq_lens, w.block_size, R)
    rows = w.num_seqs * q
    H, D = w.num_heads, w.head_size
    mx = int(w.seq_lens.max())
    parts_o = torch.empty((R, rows * H, D), dtype=torch.float32, device=DEV)
    parts_ml = torch.empty((R, rows * H, 2), dtype=torch.float32, device=DEV)
    for k, (lc, lt) in enumerate(poison_past_local_ends(shards, w.seq_lens, w.block_size, R)
                                 if poison else shards):
        n = B.paged_attn_decode_dcp_workspace_size(w.num_seqs, q, mx, R, r.p)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=DEV)
        B.paged_attn_decode_dcp_partial(parts_o[k], parts_ml[k], r.query, lc.to(DEV),
                                        lt.to(DEV), w.seq_lens.to(DEV), q, mx, R, k, r.p, ws)
    out = torch.full_like(r.query, float("nan"))
    B.paged_attn_dcp_combine(out, parts_o, parts_ml, r.p)
    assert_no_device_error(case)
    ref = O.paged_attn_decode_multi(w.query, oracle_cache_after_write(w), w.block_tables,
                                    w.seq_lens, q, oracle_params(w))
    assert_close(out, ref, case)
    # each share alone: its normalised o against the oracle's share of that rank
    op = oracle_params(w)
    for k, (lc, lt) in enumerate(shards):
        o, _, l = O.paged_attn_decode_dcp_partials(w.query, lc, lt, w.seq_lens, q, R, k, op)
        got = parts_o[k].cpu().double().view(rows, H * D)
        seen = (l > 0).repeat_interleave(D, dim=1)
        err = (got - o).abs()[seen]
        assert err.numel() == 0 or err.max().item() <= 2e-2, (k, err.max().item())
        assert torch.equal(parts_ml[k, :, 1].cpu().view(rows, H) > 0, l > 0), k


def test_dcp_decode_module_single_rank_is_plain_decode():
    w, _ = batch(207, world=1, H=32, KVH=8, lens=lens_of(7, 5, 1, 800))
    r = CudaRun(w)
    r.write()
    out = torch.full_like(r.query, float("nan"))
    DCP.dcp_decode(out, r.query, r.cache, r.tables, w.seq_lens.to(DEV), 1,
                   int(w.seq_lens.max()), r.p,
                   workspace=torch.empty(1 << 20, dtype=torch.uint8, device=DEV))
    ref = r.decode()
    assert_no_device_error("dcp module")
    assert (out.double() - ref.double()).abs().max().item() <= 2e-2
