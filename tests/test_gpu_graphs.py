"""The calls inside a CUDA graph (backends.utils AttentionCGSupport: decodes,
uniform speculative batches and mixed batches are replayed from captured
graphs).  Each call enqueues kernels only, with every argument by value or
in device memory, so a captured step replayed on new input values must give
exactly the outputs of the same calls made directly."""
import pytest
import torch

from paged_kv_cache_246_gb300 import binding as B
from paged_kv_cache_246_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_helpers import DEV, CudaRun, assert_no_device_error  # noqa: E402


def _mixed_and_spec():
    mixed = W.make_config(4, scale_down=16)      # chunked ALiBi prefill + decodes
    spec = W.make_config(9, scale_down=16)       # 8 sequences x 4 tokens
    return mixed, spec


def test_captured_step_replays_exactly():
    mixed, spec = _mixed_and_spec()
    rm, rs = CudaRun(mixed), CudaRun(spec)
    P, Tp = mixed.num_prefill_seqs, mixed.num_prefill_tokens
    q, cuq, cuk, bt, mq, mk = mixed.prefill_slices()
    cuq, cuk = cuq.to(DEV), cuk.to(DEV)
    dmax = int(mixed.seq_lens[P:].max())
    smax = int(spec.seq_lens.max())
    ws_d = torch.empty(max(B.paged_attn_decode_workspace_size(mixed.num_seqs - P, dmax, rm.p),
                           256), dtype=torch.uint8, device=DEV)
    ws_s = torch.empty(max(B.paged_attn_decode_multi_workspace_size(spec.num_seqs, 4, smax, rs.p),
                           256), dtype=torch.uint8, device=DEV)
    out_m = torch.zeros_like(rm.query)
    out_s = torch.zeros_like(rs.query)
    sl_m, sl_s = mixed.seq_lens.to(DEV), spec.seq_lens.to(DEV)
    cache_m0, cache_s0 = rm.cache.clone(), rs.cache.clone()

    def step():
        B.kv_cache_write(rm.key, rm.value, rm.cache, rm.slots, rm.p)
        B.paged_attn_prefill_varlen(out_m[:Tp], rm.query[:Tp], cuq, cuk, mq, mk, rm.cache,
                                    rm.tables[:P], rm.p)
        B.paged_attn_decode(out_m[Tp:], rm.query[Tp:], rm.cache, rm.tables[P:], sl_m[P:], dmax,
                            rm.p, ws_d)
        B.kv_cache_write(rs.key, rs.value, rs.cache, rs.slots, rs.p)
        B.paged_attn_decode_multi(out_s, rs.query, rs.cache, rs.tables, sl_s, 4, smax, rs.p, ws_s)

    step()  # first calls on this device happen outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    assert_no_device_error("capture")

    g = torch.Generator().manual_seed(5)
    for it in range(2):
        # new step inputs, written in place into the captured buffers
        for t in (rm.query, rm.key, rm.value, rs.query, rs.key, rs.value):
            t.copy_(torch.randn(t.shape, generator=g).to(t.dtype))
        rm.cache.copy_(cache_m0)
        rs.cache.copy_(cache_s0)
        out_m.zero_()
        out_s.zero_()
        graph.replay()
        torch.cuda.synchronize()
        got_m, got_s = out_m.clone(), out_s.clone()
        rm.cache.copy_(cache_m0)
        rs.cache.copy_(cache_s0)
        out_m.zero_()
        out_s.zero_()
        step()
        torch.cuda.synchronize()
        assert_no_device_error(f"replay {it}")
        assert torch.isfinite(got_m).all() and torch.isfinite(got_s).all()
        assert torch.equal(got_m, out_m), it
        assert torch.equal(got_s, out_s), it
