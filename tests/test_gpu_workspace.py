"""The decode workspace holds the split partials of one call: its contents on
entry do not matter, and one workspace serves calls of different sizes one
after another."""
import pytest
import torch

import oracle as O
from gpu_helpers import (DEV, CudaRun, assert_close, assert_no_device_error,
                         oracle_cache_after_write, oracle_params)
from paged_kv_cache_246_gb300 import binding as B
from paged_kv_cache_246_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _workload(seed, lens, multi=0, H=32, KVH=8):
    g = torch.Generator().manual_seed(seed)
    return W.build(name=f"ws{seed}", g=g, dtype=torch.bfloat16, num_heads=H, num_kv_heads=KVH,
                   head_size=128, block_size=16, seq_lens=lens,
                   query_lens=[multi or 1] * len(lens), num_prefill_seqs=0, alibi=False,
                   sliding_window=0, num_blocks=None, causal=True, multi_query_len=multi)


def _lens(seed, n, lo, hi):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


@pytest.mark.parametrize("fill", [0x00, 0x7F, 0xFF])
def test_one_workspace_across_sizes_and_contents(fill):
    # long sequences in a small batch (several splits per sequence), then a
    # batch of 4-token decodes with another split plan, on one workspace
    # whose bytes start as `fill` (0xFF: every partial a NaN)
    wa = _workload(61, _lens(61, 6, 3000, 9000))
    wb = _workload(62, _lens(62, 8, 100, 1500), multi=4)
    ra, rb = CudaRun(wa), CudaRun(wb)
    ra.write()
    rb.write()
    mxa, mxb = int(wa.seq_lens.max()), int(wb.seq_lens.max())
    na = B.paged_attn_decode_workspace_size(wa.num_seqs, mxa, ra.p)
    nb = B.paged_attn_decode_multi_workspace_size(wb.num_seqs, 4, mxb, rb.p)
    assert na > 0 and nb > 0
    ws = torch.full((max(na, nb),), fill, dtype=torch.uint8, device=DEV)

    out_a = torch.full_like(ra.query, float("nan"))
    B.paged_attn_decode(out_a, ra.query, ra.cache, ra.tables, wa.seq_lens.to(DEV), mxa, ra.p, ws)
    assert_no_device_error("first decode")
    ref_a = O.paged_attn_decode(wa.query, oracle_cache_after_write(wa), wa.block_tables,
                                wa.seq_lens, oracle_params(wa))
    assert_close(out_a, ref_a, "first decode")

    out_b = torch.full_like(rb.query, float("nan"))
    B.paged_attn_decode_multi(out_b, rb.query, rb.cache, rb.tables, wb.seq_lens.to(DEV), 4, mxb,
                              rb.p, ws)
    assert_no_device_error("multi-token decode")
    ref_b = O.paged_attn_decode_multi(wb.query, oracle_cache_after_write(wb), wb.block_tables,
                                      wb.seq_lens, 4, oracle_params(wb))
    assert_close(out_b, ref_b, "multi-token decode")

    # back to the first shape: bit for bit the first result
    again = torch.full_like(ra.query, float("nan"))
    B.paged_attn_decode(again, ra.query, ra.cache, ra.tables, wa.seq_lens.to(DEV), mxa, ra.p, ws)
    assert_no_device_error("repeat")
    assert torch.equal(again, out_a)
