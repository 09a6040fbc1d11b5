"""GPU parity at the full workload sizes, in the launch configuration the
bench times: every cache write and block move compared whole and bit-exact;
attention compared on sampled sequences / rows the oracle computes one by
one (first, last, longest, shortest, tile and split boundaries, random)."""
import pytest
import torch

import oracle as O
from paged_kv_cache_246_gb300 import binding as B
from paged_kv_cache_246_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_helpers import (DEV, CudaRun, assert_close, assert_no_device_error,  # noqa: E402
                             oracle_params)


def _sample_seqs(seq_lens, n_random=6, seed=0):
    L = seq_lens.tolist()
    picks = {0, len(L) - 1, L.index(max(L)), L.index(min(L))}
    g = torch.Generator().manual_seed(seed)
    picks |= set(torch.randint(0, len(L), (n_random,), generator=g).tolist())
    return sorted(picks)


def _sample_rows(cu_q, per_seq=3, seed=0):
    g = torch.Generator().manual_seed(seed)
    rows = set()
    cu = cu_q.tolist()
    for b in range(len(cu) - 1):
        a, e = cu[b], cu[b + 1]
        if e <= a:
            continue
        rows |= {a, e - 1, min(e - 1, a + 127), min(e - 1, a + 128)}
        rows |= set(torch.randint(a, e, (per_seq,), generator=g).tolist())
    return sorted(rows)


def _write_and_check(w, r):
    r.write()
    assert_no_device_error(w.name + " write")
    ref = w.kv_cache  # the oracle writes in place on the CPU copy
    O.kv_cache_write(w.key, w.value, ref, w.slot_mapping, oracle_params(w))
    assert torch.equal(r.cache.cpu().view(torch.int16), ref.view(torch.int16))
    return ref


def test_llama3_8b_decode_full():
    w = W.make_config(2)
    r = CudaRun(w)
    ref_cache = _write_and_check(w, r)
    out = r.decode()
    assert_no_device_error("decode")
    seqs = _sample_seqs(w.seq_lens)
    ref = O.paged_attn_decode(w.query, ref_cache, w.block_tables, w.seq_lens,
                              oracle_params(w), seqs=seqs)
    assert_close(out[seqs], ref[seqs], "llama3_8b_decode")


def test_varlen_prefill_full():
    w = W.make_config(3)
    r = CudaRun(w)
    ref_cache = _write_and_check(w, r)
    out = r.prefill()
    assert_no_device_error("prefill")
    q, cuq, cuk, bt, _, _ = w.prefill_slices()
    rows = _sample_rows(cuq)
    ref = O.paged_attn_prefill_varlen(q, cuq, cuk, ref_cache, bt, oracle_params(w), rows=rows)
    assert_close(out[rows], ref[rows], "varlen_prefill")


def test_encoder_varlen_prefill_full():
    w = W.make_config(6)
    r = CudaRun(w)
    ref_cache = _write_and_check(w, r)
    out = r.prefill()
    assert_no_device_error("encoder prefill")
    q, cuq, cuk, bt, _, _ = w.prefill_slices()
    rows = _sample_rows(cuq, per_seq=2)
    ref = O.paged_attn_prefill_varlen(q, cuq, cuk, ref_cache, bt, oracle_params(w), rows=rows)
    assert_close(out[rows], ref[rows], "encoder_varlen_prefill")


def test_llama3_8b_decode_fp8_full():
    w = W.make_config(7)
    r = CudaRun(w)
    ref_cache = _write_and_check(w, r)
    out = r.decode()
    assert_no_device_error("fp8 decode")
    seqs = _sample_seqs(w.seq_lens)
    ref = O.paged_attn_decode(w.query, ref_cache, w.block_tables, w.seq_lens,
                              oracle_params(w), seqs=seqs)
    assert_close(out[seqs], ref[seqs], "llama3_8b_decode_fp8")


def test_varlen_prefill_fp8_full():
    w = W.make_config(8)
    r = CudaRun(w)
    ref_cache = _write_and_check(w, r)
    out = r.prefill()
    assert_no_device_error("fp8 prefill")
    q, cuq, cuk, bt, _, _ = w.prefill_slices()
    rows = _sample_rows(cuq, per_seq=2)
    ref = O.paged_attn_prefill_varlen(q, cuq, cuk, ref_cache, bt, oracle_params(w), rows=rows)
    assert_close(out[rows], ref[rows], "varlen_prefill_fp8")


def test_llama3_8b_spec_decode_full():
    w = W.make_config(9)
    r = CudaRun(w)
    ref_cache = _write_and_check(w, r)
    out = r.decode_multi()
    assert_no_device_error("spec decode")
    seqs = _sample_seqs(w.seq_lens)
    ref = O.paged_attn_decode_multi(w.query, ref_cache, w.block_tables, w.seq_lens,
                                    w.multi_query_len, oracle_params(w), seqs=seqs)
    q = w.multi_query_len
    rows = [b * q + t for b in seqs for t in range(q)]
    assert_close(out[rows], ref[rows], "llama3_8b_spec_decode")


def test_mixed_chunked_alibi_full():
    w = W.make_config(4)
    r = CudaRun(w)
    ref_cache = _write_and_check(w, r)
    pre = r.prefill()
    dec = r.decode()
    assert_no_device_error("mixed")
    op = oracle_params(w)
    q, cuq, cuk, bt, _, _ = w.prefill_slices()
    rows = _sample_rows(cuq, per_seq=2)
    ref = O.paged_attn_prefill_varlen(q, cuq, cuk, ref_cache, bt, op, rows=rows)
    assert_close(pre[rows], ref[rows], "mixed prefill")
    dq, dbt, dsl, _ = w.decode_slices()
    seqs = _sample_seqs(dsl)
    refd = O.paged_attn_decode(dq, ref_cache, dbt, dsl, op, seqs=seqs)
    assert_close(dec[seqs], refd[seqs], "mixed decode")


def test_swa_long_decode_and_block_ops_full():
    w = W.make_config(5)
    r = CudaRun(w)
    ref_cache = _write_and_check(w, r)
    out = r.decode()
    assert_no_device_error("swa decode")
    seqs = _sample_seqs(w.seq_lens, n_random=3)
    ref = O.paged_attn_decode(w.query, ref_cache, w.block_tables, w.seq_lens,
                              oracle_params(w), seqs=seqs)
    assert_close(out[seqs], ref[seqs], "swa decode")

    # copy_blocks: 2048 pairs
    B.kv_copy_blocks([r.cache], w.copy_pairs.to(DEV), r.p)
    assert_no_device_error("copy")
    O.kv_copy_blocks([ref_cache], w.copy_pairs.tolist())
    assert torch.equal(r.cache.cpu().view(torch.int16), ref_cache.view(torch.int16))

    # swap 4096 blocks out to pinned host memory and back
    n = w.swap_pairs.shape[0]
    host = torch.empty((2, n, w.kv_cache.shape[2]), dtype=w.dtype).pin_memory()
    B.kv_swap_blocks(r.cache, host, w.swap_pairs, r.p)
    torch.cuda.synchronize()
    src = w.swap_pairs[:, 0]
    assert torch.equal(host.view(torch.int16), ref_cache[:, src].view(torch.int16))
    r.cache[:, src.to(DEV)] = 0
    B.kv_swap_blocks(host, r.cache, w.swap_pairs[:, [1, 0]].contiguous(), r.p)
    assert_no_device_error("swap")
    assert torch.equal(r.cache.cpu().view(torch.int16), ref_cache.view(torch.int16))
