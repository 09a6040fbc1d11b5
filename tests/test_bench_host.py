"""Host-side arithmetic of bench.py (no GPU): the algorithmic bytes and flops
behind every roofline number, checked against closed forms, and the guard
that drops a profiled DRAM traffic figure once the kernel source changed."""
import hashlib
import json
import os

import pytest
import torch

import bench
from paged_kv_cache_246_gb300 import workloads as W


def _decode_workload(lens, window=0, mq=0, fp8=False):
    g = torch.Generator().manual_seed(7)
    q = mq or 1
    extra = dict(kv_cache_dtype="fp8_e4m3", k_scale=0.02, v_scale=0.02) if fp8 else {}
    return W.build(name="t", g=g, dtype=torch.bfloat16, num_heads=8, num_kv_heads=2,
                   head_size=64, block_size=16, seq_lens=lens, query_lens=[q] * len(lens),
                   num_prefill_seqs=0, alibi=False, sliding_window=window,
                   multi_query_len=mq, **extra)


def test_decode_bytes_closed_form():
    lens = [1, 17, 300]
    w = _decode_workload(lens)
    dec_bytes, flops = bench.algorithmic(w)
    row = 2 * 64                                        # KVH * D
    kv = sum(lens) * row * 2 * 2                        # K and V, 2-byte elements
    qo = len(lens) * 8 * 64 * 2 * 2                     # query in, output out
    assert dec_bytes == kv + qo and flops == 0


def test_decode_bytes_window_multi_and_fp8():
    lens = [5, 100, 900]
    w = _decode_workload(lens, window=64, mq=4, fp8=True)
    dec_bytes, _ = bench.algorithmic(w)
    # each sequence's 4 tokens see the last 64 + 3 keys at most; 1-byte codes
    keys = sum(min(L, 64 + 3) for L in lens)
    assert dec_bytes == keys * 2 * 64 * 1 * 2 + len(lens) * 4 * 8 * 64 * 2 * 2


def test_prefill_flops_closed_form():
    g = torch.Generator().manual_seed(3)
    # causal prompt of n tokens: n (n + 1) / 2 visible pairs; a chunk of q
    # tokens over c cached ones: q c + q (q + 1) / 2; encoder: q L
    n, c, q = 37, 50, 20
    for causal, lens, qlens, pairs in (
            (True, [n], [n], n * (n + 1) // 2),
            (True, [c + q], [q], q * c + q * (q + 1) // 2),
            (False, [c + q], [q], q * (c + q))):
        w = W.build(name="p", g=g, dtype=torch.bfloat16, num_heads=4, num_kv_heads=2,
                    head_size=64, block_size=16, seq_lens=lens, query_lens=qlens,
                    num_prefill_seqs=1, alibi=False, sliding_window=0, causal=causal)
        _, flops = bench.algorithmic(w)
        assert flops == 4 * 4 * 64 * pairs, (causal, lens, qlens)


def test_prefill_footprint_states_the_bytes():
    w = W.make_config(3)
    text = bench.prefill_footprint(w)
    tq = int(w.query_lens.sum())
    assert f"{tq * 32 * 128 * 2 * 2 / 1e6:.0f} MB" in text and "larger than L2" in text


def test_profiled_traffic_needs_the_captured_source(tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_cache_246_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "k.md").write_text(
        f"# k\n\nsource_sha256_16: {digest}  (k.cu)\ntraffic_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "HERE", str(tmp_path))
    assert bench.profiled_traffic("k.cu", "k.md") == 12345
    src.write_bytes(b"__global__ void k() { }\n")      # any edit after the capture
    assert bench.profiled_traffic("k.cu", "k.md") is None
    assert bench.profiled_traffic("missing.cu", "k.md") is None


def test_every_profiled_workload_names_a_committed_summary():
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for cfg, (src, summary) in bench.PROFILE_OF.items():
        assert os.path.exists(os.path.join(here, "paged_kv_cache_246_gb300", "csrc", src)), cfg
        assert os.path.exists(os.path.join(here, "profiles", summary)), cfg


def test_write_bytes_closed_form():
    lens = [3, 40]
    for fp8, out_el in ((False, 2), (True, 1)):
        w = _decode_workload(lens, fp8=fp8)
        # 2 new tokens: K and V rows of 2 x 64 elements, read as bf16, written
        # in the cache's element size
        assert bench.write_bytes(w) == 2 * 2 * 2 * 64 * (2 + out_el)


def test_extra_workloads_default_and_list():
    class A:
        extra, workload, scale_down = "auto", "decode", 1
    assert bench.extra_workloads(A) == ["prefill", "mixed", "swa"]
    A.workload = "prefill"
    assert bench.extra_workloads(A) == []
    A.extra = "swa,spec_decode"
    assert bench.extra_workloads(A) == ["swa", "spec_decode"]
    A.extra = "none"
    assert bench.extra_workloads(A) == []
    A.extra = "bogus"
    with pytest.raises(SystemExit):
        bench.extra_workloads(A)


def test_reference_line_uses_the_gpu_arms_config_and_affinity_cores(monkeypatch, capsys):
    # the tiny decode stands in for the headline workload to keep this quick
    monkeypatch.setitem(bench.CFG_OF, "decode", 1)

    class A:
        workload, steps, warmup, gpus = "decode", 1, 3, 1
    line = bench.run_reference(A, 1, 0)
    printed = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert printed == json.loads(json.dumps(line))
    assert line["config"] == bench.config_of(W.make_config(1), 1, 1)
    assert line["impl"] == "reference" and line["value"] > 0
    cpu = line["cpu_baseline"]
    assert cpu["cores"] == len(os.sched_getaffinity(0)) and cpu["value_1core"] > 0
