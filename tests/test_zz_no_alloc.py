"""paged_attn_decode_noalloc: decode for callers that may not allocate device
memory (for instance a plugin that only receives buffers from its host
framework).  Its split partials live in the library's static device scratch
instead of a caller workspace; its output must equal paged_attn_decode with a
workspace bit for bit, call after call, match the oracle, and it must not
allocate.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test."""
import pytest
import torch

import oracle as O
from paged_kv_cache_246_gb300 import binding as B
from paged_kv_cache_246_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_helpers import (DEV, CudaRun, assert_close, assert_no_device_error,  # noqa: E402
                             oracle_cache_after_write, oracle_params)


def _allocations():
    return torch.cuda.memory_stats(DEV).get("allocation.all.allocated", 0)


@pytest.mark.parametrize("cfg,scale_down", [(2, 4), (5, 4), (1, 1)])
def test_noalloc_matches_workspace_decode_twice(cfg, scale_down):
    w = W.make_config(cfg, scale_down=scale_down)
    r = CudaRun(w)
    r.write()
    ref = r.decode()                       # existing entry point, torch workspace
    assert_no_device_error("reference decode")
    mx = int(w.seq_lens.max())
    need = B.paged_attn_decode_workspace_size(w.num_seqs, mx, r.p)
    assert need <= B.PKV_DECODE_STATIC_SCRATCH_BYTES
    if cfg != 1:
        assert need > 0                    # the split pass and the combine both run

    # the same rows against the oracle directly (a sample of the sequences)
    seqs = sorted({0, w.num_seqs // 2, w.num_seqs - 1})
    want = O.paged_attn_decode(w.query, oracle_cache_after_write(w), w.block_tables, w.seq_lens,
                               oracle_params(w), seqs=seqs)

    lens = w.seq_lens.to(DEV)
    # another decode that fills the scratch with different partials: every
    # sequence at the longest length (its table's unused entries name block
    # 0, a valid block) and other queries
    other_lens = torch.full_like(lens, mx)
    other_q = torch.randn(r.query.shape, generator=torch.Generator().manual_seed(5)).to(
        device=DEV, dtype=r.query.dtype)
    other_out = torch.empty_like(r.query)
    out = torch.empty_like(r.query)
    for call in range(2):                  # two calls in a row share the scratch
        if call == 1:
            B.paged_attn_decode_noalloc(other_out, other_q, r.cache, r.tables, other_lens, mx,
                                        r.p)
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free_before, allocs_before = torch.cuda.mem_get_info(DEV)[0], _allocations()
        B.paged_attn_decode_noalloc(out, r.query, r.cache, r.tables, lens, mx, r.p)
        torch.cuda.synchronize()
        assert _allocations() == allocs_before
        if call == 1:                      # after the one-time set-up: nothing allocated
            assert torch.cuda.mem_get_info(DEV)[0] == free_before
        assert_no_device_error(f"noalloc call {call}")
        assert torch.equal(out, ref), f"call {call}: differs from the workspace decode"
        assert_close(out[seqs], want[seqs], f"noalloc call {call} vs oracle")


def test_noalloc_rejects_sizes_beyond_the_scratch():
    w = W.make_config(1)
    r = CudaRun(w)
    big_seqs, big_len = 4096, 65536
    assert B.paged_attn_decode_workspace_size(big_seqs, big_len, r.p) > \
        B.PKV_DECODE_STATIC_SCRATCH_BYTES
    out = torch.empty(big_seqs, w.num_heads * w.head_size, dtype=w.dtype, device=DEV)
    q = torch.zeros_like(out)
    tables = torch.zeros(big_seqs, 1, dtype=torch.int32, device=DEV)
    lens = torch.ones(big_seqs, dtype=torch.int32, device=DEV)
    with pytest.raises(B.PkvError) as e:
        B.paged_attn_decode_noalloc(out, q, r.cache, tables, lens, big_len, r.p)
    assert e.value.status == B.PKV_ERR_UNSUPPORTED
