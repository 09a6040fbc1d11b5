"""Shared helpers of the GPU parity tests: run a Workload through the C ABI
and through the fp64 oracle on the same bits, and compare."""
from __future__ import annotations

import torch

import oracle as O
from paged_kv_cache_246_gb300 import binding as B
from paged_kv_cache_246_gb300 import workloads as W

# Attention tolerance on fp16/bf16 outputs with fp32 accumulation.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3

DEV = torch.device("cuda:0")


def oracle_params(w: W.Workload) -> O.AttnParams:
    return O.AttnParams(w.num_heads, w.num_kv_heads, w.head_size, w.block_size, w.scale,
                        None if w.alibi_slopes is None else w.alibi_slopes.tolist(),
                        w.sliding_window, w.causal, w.kv_cache_dtype, w.k_scale, w.v_scale)


class CudaRun:
    """Device copies of a workload plus the library's params."""

    def __init__(self, w: W.Workload):
        self.w = w
        self.slopes = None if w.alibi_slopes is None else w.alibi_slopes.to(DEV)
        self.p = B.make_params(w.num_heads, w.num_kv_heads, w.head_size, w.block_size, w.dtype,
                               w.scale, self.slopes, w.sliding_window, not w.causal,
                               w.kv_cache_dtype, w.k_scale, w.v_scale)
        self.cache = w.kv_cache.to(DEV)
        self.key = w.key.to(DEV)
        self.value = w.value.to(DEV)
        self.slots = w.slot_mapping.to(DEV)
        self.query = w.query.to(DEV)
        self.tables = w.block_tables.to(DEV)

    def write(self):
        B.kv_cache_write(self.key, self.value, self.cache, self.slots, self.p)

    def decode(self, max_seq_len=None):
        w = self.w
        P, Tp = w.num_prefill_seqs, w.num_prefill_tokens
        q = self.query[Tp:]
        bt = self.tables[P:]
        sl = w.seq_lens[P:].to(DEV)
        mx = int(w.seq_lens[P:].max()) if max_seq_len is None else max_seq_len
        out = torch.full_like(q, float("nan"))
        n = B.paged_attn_decode_workspace_size(q.shape[0], mx, self.p)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
        B.paged_attn_decode(out, q, self.cache, bt, sl, mx, self.p, ws)
        return out

    def decode_multi(self, max_seq_len=None):
        """Every sequence decodes w.multi_query_len tokens (rows b * q + t)."""
        w = self.w
        q = w.multi_query_len
        sl = w.seq_lens.to(DEV)
        mx = int(w.seq_lens.max()) if max_seq_len is None else max_seq_len
        out = torch.full_like(self.query, float("nan"))
        n = B.paged_attn_decode_multi_workspace_size(w.num_seqs, q, mx, self.p)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
        B.paged_attn_decode_multi(out, self.query, self.cache, self.tables, sl, q, mx, self.p, ws)
        return out

    def prefill(self):
        q, cuq, cuk, bt, mq, mk = self.w.prefill_slices()
        Tp = q.shape[0]
        out = torch.full_like(self.query[:Tp], float("nan"))
        B.paged_attn_prefill_varlen(out, self.query[:Tp], cuq.to(DEV), cuk.to(DEV), mq, mk,
                                    self.cache, self.tables[:bt.shape[0]], self.p)
        return out


def oracle_cache_after_write(w: W.Workload) -> torch.Tensor:
    ref = w.kv_cache.clone()
    O.kv_cache_write(w.key, w.value, ref, w.slot_mapping, oracle_params(w))
    return ref


def assert_close(got: torch.Tensor, ref: torch.Tensor, what: str):
    got = got.detach().cpu().double()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert torch.isfinite(got).all(), f"{what}: non-finite output"
    err = (got - ref).abs()
    mx, mean = err.max().item(), err.mean().item()
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def assert_no_device_error(where: str):
    torch.cuda.synchronize()
    st, d = B.device_error()
    assert st == B.PKV_OK, f"{where}: device error {B.status_string(st)} at {d}"
