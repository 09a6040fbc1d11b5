"""paged_attn_decode_noalloc: decode for callers that may not allocate device
memory (for instance a plugin that only receives buffers from its host
framework).  Its split partials live in the library's static device scratch
instead of a caller workspace; its output must match paged_attn_decode with a
workspace, call after call, and it must not allocate.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test."""
import pytest
import torch

from paged_kv_cache_246_gb300 import binding as B
from paged_kv_cache_246_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_helpers import DEV, CudaRun, assert_no_device_error  # noqa: E402

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def _noalloc(r, out):
    w = r.w
    B.paged_attn_decode_noalloc(out, r.query, r.cache, r.tables, w.seq_lens.to(DEV),
                                int(w.seq_lens.max()), r.p)


@pytest.mark.parametrize("cfg,scale_down", [(2, 2), (5, 4), (1, 1)])
def test_noalloc_matches_workspace_decode_twice(cfg, scale_down):
    w = W.make_config(cfg, scale_down=scale_down)
    r = CudaRun(w)
    r.write()
    ref = r.decode().double()             # existing entry point, torch workspace
    assert_no_device_error("reference decode")
    need = B.paged_attn_decode_workspace_size(w.num_seqs, int(w.seq_lens.max()), r.p)
    assert need <= 64 << 20
    out = torch.empty_like(r.query)
    for call in range(2):                  # two calls in a row share the scratch
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        _noalloc(r, out)
        torch.cuda.synchronize()
        if call == 1:                      # after set-up: nothing allocated
            assert torch.cuda.mem_get_info()[0] == free_before
        assert_no_device_error(f"noalloc call {call}")
        err = (out.double() - ref).abs()
        assert torch.isfinite(out).all()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (
            call, err.max().item(), err.mean().item())


def test_noalloc_rejects_sizes_beyond_the_scratch():
    w = W.make_config(1)
    r = CudaRun(w)
    big_seqs, big_len = 4096, 65536
    assert B.paged_attn_decode_workspace_size(big_seqs, big_len, r.p) > 64 << 20
    out = torch.empty(big_seqs, w.num_heads * w.head_size, dtype=w.dtype, device=DEV)
    q = torch.zeros_like(out)
    tables = torch.zeros(big_seqs, 1, dtype=torch.int32, device=DEV)
    lens = torch.ones(big_seqs, dtype=torch.int32, device=DEV)
    with pytest.raises(B.PkvError) as e:
        B.paged_attn_decode_noalloc(out, q, r.cache, tables, lens, big_len, r.p)
    assert e.value.status == B.PKV_ERR_UNSUPPORTED
