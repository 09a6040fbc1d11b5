"""Benchmark of the paged-KV attention path on GB300.

Headline workload: the Llama-3-8B-shaped decode step (bf16, 256 sequences,
32 query / 8 KV heads, head 128, block 16, seq_len ~ U[512, 4096], pool =
needed blocks + 10%, tables randomly permuted).  One step = kv_cache_write of
the 256 new tokens, then paged_attn_decode (split-KV pass, and the combine
when a sequence is split).

Beside it the default run measures, each with its own warm-up, timed steps
and clock record, and reports in the line's ``workloads`` object:
  varlen_prefill       16 causal prompts, log-uniform [128, 8192]: the write
                       of all prompt tokens, then paged_attn_prefill_varlen
                       (TFLOP/s against the bf16 tensor peak)
  mixed_chunked_alibi  8 ALiBi prefill chunks over cached context, then 192
                       decodes (prefill TFLOP/s and decode GB/s)
  swa_long_decode      64 sequences of 16k-32k tokens under a 4096-token
                       window (decode GB/s), then kv_copy_blocks of 2048
                       pairs (HBM) and kv_swap_blocks of 4096 blocks out to
                       pinned host memory and back (against a same-size
                       pinned copy)
Every record carries the cache write on its own (microseconds and GB/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode|prefill|mixed|swa|encoder|decode_fp8|prefill_fp8|
                              spec_decode|dcp2_share] [--extra auto|none|a,b,...]

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own
replica of the workload on its own GPU (the path has no exchange step), so
scaling is weak and `value` counts the tokens of all ranks.
--impl reference times the fp64 CPU oracle on this host's cores instead.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

from paged_kv_cache_246_gb300 import workloads as W  # noqa: E402

METRIC = ("decode tokens/s and HBM GB/s (%peak); prefill TFLOP/s (%bf16 peak), 1×GB300")
# committed ncu summary (kernel source, file) per workload: DRAM traffic per launch
PROFILE_OF = {2: ("decode.cu", "decode_kernel_llama3_8b_decode.md"),
              3: ("prefill.cu", "prefill_tc_kernel_varlen_prefill.md"),
              4: ("decode.cu", "decode_kernel_mixed_chunked_alibi.md"),
              5: ("decode.cu", "decode_kernel_swa_long_decode.md"),
              7: ("decode.cu", "decode_kernel_llama3_8b_decode_fp8.md"),
              8: ("prefill.cu", "prefill_tc_kernel_varlen_prefill_fp8.md"),
              9: ("decode.cu", "decode_kernel_llama3_8b_spec_decode.md")}
CFG_OF = {"decode": 2, "prefill": 3, "mixed": 4, "swa": 5, "encoder": 6, "decode_fp8": 7,
          "prefill_fp8": 8, "spec_decode": 9, "dcp2_share": 2}


def peaks():
    try:
        with open(os.path.join(HERE, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(
            d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = list(csv.reader(io.StringIO(out)))
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the workload on the device
# ---------------------------------------------------------------------------
class Step:
    """Device-resident tensors of one workload and the calls of one step."""

    def __init__(self, w: W.Workload, dev, B):
        self.w, self.B, self.dev = w, B, dev
        self.slopes = None if w.alibi_slopes is None else w.alibi_slopes.to(dev)
        self.p = B.make_params(w.num_heads, w.num_kv_heads, w.head_size, w.block_size, w.dtype,
                               w.scale, self.slopes, w.sliding_window, not w.causal,
                               w.kv_cache_dtype, w.k_scale, w.v_scale)
        self.cache = w.kv_cache.to(dev)
        self.key, self.value = w.key.to(dev), w.value.to(dev)
        self.slots = w.slot_mapping.to(dev)
        self.query = w.query.to(dev)
        self.tables = w.block_tables.to(dev)
        self.seq_lens = w.seq_lens.to(dev)
        self.out = torch.empty_like(self.query)
        P, Tp = w.num_prefill_seqs, w.num_prefill_tokens
        self.P, self.Tp = P, Tp
        self.has_prefill = P > 0
        self.has_decode = w.num_seqs > P
        if self.has_prefill:
            q, cuq, cuk, bt, mq, mk = w.prefill_slices()
            self.cuq, self.cuk, self.mq, self.mk = cuq.to(dev), cuk.to(dev), mq, mk
        self.mq_len = w.multi_query_len
        if self.has_decode:
            self.dmax = int(w.seq_lens[P:].max())
            if self.mq_len:
                n = B.paged_attn_decode_multi_workspace_size(w.num_seqs, self.mq_len, self.dmax,
                                                             self.p)
            else:
                n = B.paged_attn_decode_workspace_size(w.num_seqs - P, self.dmax, self.p)
            self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
            self.multi_split = n > 0
        self.ev = []

    def launches_per_step(self) -> int:
        n = 1
        if self.has_prefill:
            n += 1
        if self.has_decode:
            n += 2 if self.multi_split else 1
        return n

    def run(self, mark=False):
        B = self.B
        if mark:
            ew = torch.cuda.Event(enable_timing=True)
            ew.record()
        B.kv_cache_write(self.key, self.value, self.cache, self.slots, self.p)
        if mark:
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record()
        if self.has_prefill:
            B.paged_attn_prefill_varlen(self.out[:self.Tp], self.query[:self.Tp], self.cuq,
                                        self.cuk, self.mq, self.mk, self.cache,
                                        self.tables[:self.P], self.p)
        if mark:
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record()
        if self.has_decode and self.mq_len:
            B.paged_attn_decode_multi(self.out, self.query, self.cache, self.tables,
                                      self.seq_lens, self.mq_len, self.dmax, self.p, self.ws)
        elif self.has_decode:
            B.paged_attn_decode(self.out[self.Tp:], self.query[self.Tp:], self.cache,
                                self.tables[self.P:], self.seq_lens[self.P:], self.dmax, self.p,
                                self.ws)
        if mark:
            e2 = torch.cuda.Event(enable_timing=True)
            e2.record()
            self.ev.append((ew, e0, e1, e2))


def algorithmic(w: W.Workload):
    """Bytes read+written by the decode call and flops of the prefill call."""
    P = w.num_prefill_seqs
    el = 2
    kv_el = 1 if w.kv_cache_dtype == "fp8_e4m3" else 2   # cache bytes per element
    row = w.num_kv_heads * w.head_size
    dec_bytes = 0
    mq = max(1, w.multi_query_len)   # query tokens per decoding sequence
    for L in w.seq_lens[P:].tolist():
        # keys visible to any of the sequence's query tokens
        keys = min(L, w.sliding_window + mq - 1) if w.sliding_window > 0 else L
        dec_bytes += keys * row * kv_el * 2       # K and V of every visible token
    nd = w.num_seqs - P
    dec_bytes += nd * mq * w.num_heads * w.head_size * el * 2   # query in, output out
    flops = 0
    for q, L in zip(w.query_lens[:P].tolist(), w.seq_lens[:P].tolist()):
        c = L - q
        pairs = 0
        for t in range(q):      # keys visible to query row t
            i = c + t
            if not w.causal:
                pairs += L      # encoder attention: the whole sequence
                continue
            lo = max(0, i - w.sliding_window + 1) if w.sliding_window > 0 else 0
            pairs += i - lo + 1
        flops += 4 * w.num_heads * w.head_size * pairs   # q.k and p.V
    return dec_bytes, flops


def prefill_footprint(w: W.Workload) -> str:
    """The L2 statement of a prefill-only step: what one step touches."""
    P = w.num_prefill_seqs
    tq = int(w.query_lens[:P].sum())
    q_bytes = tq * w.num_heads * w.head_size * 2 * 2          # queries in, output out
    kv_el = 1 if w.kv_cache_dtype == "fp8_e4m3" else 2
    kv_bytes = int(w.seq_lens[:P].sum()) * w.num_kv_heads * w.head_size * kv_el * 2
    return (f"no flush: inputs larger than L2 (queries + output {q_bytes / 1e6:.0f} MB, "
            f"K/V {kv_bytes / 1e6:.0f} MB per step)")


def profiled_traffic(kernel_src: str, summary: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source has changed since the capture."""
    import hashlib
    try:
        src = os.path.join(HERE, "paged_kv_cache_246_gb300", "csrc", kernel_src)
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        fields = {}
        for line in open(os.path.join(HERE, "profiles", summary)):
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.split()[0] if v.split() else ""
        if fields.get("source_sha256_16") != digest:
            return None
        return int(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


def step_io_bytes(st: Step):
    h2d = sum(t.numel() * t.element_size() for t in
              (st.query, st.key, st.value, st.slots, st.tables, st.seq_lens))
    if st.has_prefill:
        h2d += (st.cuq.numel() + st.cuk.numel()) * 4
    d2h = st.out.numel() * st.out.element_size()
    return h2d, d2h


def time_block_moves(st: Step, w: W.Workload, B, args, hbm: float):
    """kv_copy_blocks and kv_swap_blocks of the workload, timed apart from the
    step with CUDA events: copy against the HBM roofline (read + write
    bytes) and against a same-size contiguous device copy measured here
    (the ceiling for a move this short), swap out / in against a same-size
    contiguous pinned copy in the same direction (the host link)."""
    stream = torch.cuda.current_stream()
    block_bytes = 2 * w.kv_cache.shape[2] * w.kv_cache.element_size()   # K and V of one block
    n_copy, n_swap = int(w.copy_pairs.shape[0]), int(w.swap_pairs.shape[0])
    pairs_dev = w.copy_pairs.to(st.dev)
    host = torch.empty((2, n_swap, w.kv_cache.shape[2]), dtype=w.dtype).pin_memory()
    out_pairs = w.swap_pairs.contiguous()
    in_pairs = w.swap_pairs[:, [1, 0]].contiguous()
    flat_dev = torch.empty(n_swap * block_bytes, dtype=torch.uint8, device=st.dev)
    flat_host = torch.empty(n_swap * block_bytes, dtype=torch.uint8).pin_memory()
    flat_a = torch.ones(n_copy * block_bytes, dtype=torch.uint8, device=st.dev)
    flat_b = torch.empty_like(flat_a)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    reps = max(5, min(args.steps, 50))
    copy_ms = timed(lambda: B.kv_copy_blocks([st.cache], pairs_dev, st.p), reps)
    dev_copy_ms = timed(lambda: flat_b.copy_(flat_a), reps)
    out_ms = timed(lambda: B.kv_swap_blocks(st.cache, host, out_pairs, st.p), reps)
    in_ms = timed(lambda: B.kv_swap_blocks(host, st.cache, in_pairs, st.p), reps)
    link_out_ms = timed(lambda: flat_host.copy_(flat_dev, non_blocking=True), reps)
    link_in_ms = timed(lambda: flat_dev.copy_(flat_host, non_blocking=True), reps)
    B.check_device_error("block moves")
    copy_gbs = 2 * n_copy * block_bytes / (copy_ms * 1e-3) / 1e9
    dev_copy_gbs = 2 * n_copy * block_bytes / (dev_copy_ms * 1e-3) / 1e9
    swap_bytes = n_swap * block_bytes
    gbs = lambda ms: swap_bytes / (ms * 1e-3) / 1e9
    return {"copy_blocks": {"pairs": n_copy, "ms": copy_ms, "gbs": copy_gbs,
                            "frac_of_hbm": copy_gbs / hbm,
                            "same_size_copy_gbs": dev_copy_gbs,
                            "frac_of_same_size_copy": copy_gbs / dev_copy_gbs},
            "swap_out": {"blocks": n_swap, "ms": out_ms, "gbs": gbs(out_ms),
                         "link_gbs": gbs(link_out_ms), "frac_of_link": link_out_ms / out_ms},
            "swap_in": {"blocks": n_swap, "ms": in_ms, "gbs": gbs(in_ms),
                        "link_gbs": gbs(link_in_ms), "frac_of_link": link_in_ms / in_ms}}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline; never the target)
# ---------------------------------------------------------------------------
def host_cores() -> int:
    """Cores this process may run on (its CPU affinity)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rate(w: W.Workload, budget_s: float, threads: int | None = None):
    """Oracle throughput on a bounded sample of the workload: decode
    sequences (tokens/s) or prefill query rows (TFLOP/s-equivalent rows/s).
    ``threads``: torch intra-op threads for the oracle's fp64 tensor ops
    (None keeps the current setting); restored afterwards."""
    prev = torch.get_num_threads()
    if threads:
        torch.set_num_threads(threads)
    try:
        r = _oracle_rate(w, budget_s)
        r["threads"] = torch.get_num_threads()
        return r
    finally:
        torch.set_num_threads(prev)


def _oracle_rate(w: W.Workload, budget_s: float):
    import oracle as O
    op = O.AttnParams(w.num_heads, w.num_kv_heads, w.head_size, w.block_size, w.scale,
                      None if w.alibi_slopes is None else w.alibi_slopes.tolist(),
                      w.sliding_window, w.causal, w.kv_cache_dtype, w.k_scale, w.v_scale)
    ref = w.kv_cache.clone()
    P = w.num_prefill_seqs
    t0 = time.perf_counter()
    O.kv_cache_write(w.key, w.value, ref, w.slot_mapping, op)
    t_write = time.perf_counter() - t0
    done, t_attn = 0, 0.0
    if w.num_seqs > P:
        q, bt, sl, _ = w.decode_slices()
        nseq = sl.numel()
        mq = max(1, w.multi_query_len)
        order = torch.randperm(nseq, generator=torch.Generator().manual_seed(0)).tolist()
        for b in order:
            t1 = time.perf_counter()
            if w.multi_query_len:
                O.paged_attn_decode_multi(q, ref, bt, sl, mq, op, seqs=[b])
            else:
                O.paged_attn_decode(q, ref, bt, sl, op, seqs=[b])
            t_attn += time.perf_counter() - t1
            done += 1
            if t_attn > budget_s:
                break
        per_seq = t_attn / done
        step_s = t_write + per_seq * nseq
        return {"value": nseq * mq / step_s, "unit": "tokens/s",
                "sample": f"kv_cache_write of all {w.key.shape[0]} tokens + decode of {done} of "
                          f"{nseq} sequences (random order), scaled to the full step",
                "step_s": step_s}
    q, cuq, cuk, bt, _, _ = w.prefill_slices()
    _, flops = algorithmic(w)
    rows = torch.randperm(q.shape[0], generator=torch.Generator().manual_seed(0)).tolist()
    t1 = time.perf_counter()
    n = 0
    for k in range(0, len(rows), 8):
        O.paged_attn_prefill_varlen(q, cuq, cuk, ref, bt, op, rows=rows[k:k + 8])
        n = k + 8
        if time.perf_counter() - t1 > budget_s:
            break
    frac = min(n, len(rows)) / len(rows)
    step_s = t_write + (time.perf_counter() - t1) / frac
    return {"value": flops / step_s / 1e12, "unit": "TFLOP/s",
            "sample": f"kv_cache_write of all tokens + {min(n, len(rows))} of {len(rows)} query "
                      f"rows (random), scaled to the full step", "step_s": step_s}


def cpu_baseline(w: W.Workload, budget_s: float) -> dict:
    """The oracle on every core of this process's affinity, then on one core
    (each a bounded sample of the same step)."""
    cores = host_cores()
    full = oracle_rate(w, budget_s, threads=cores)
    one = oracle_rate(w, budget_s, threads=1)
    return {"value": full["value"], "unit": full["unit"], "cores": cores, "kind": "oracle",
            "sample": full["sample"], "threads": full["threads"],
            "value_1core": one["value"], "sample_1core": one["sample"]}


def config_of(w: W.Workload, cfg: int, world: int) -> dict:
    """The ``config`` object of a line: the same for both arms."""
    dec_bytes, _ = algorithmic(w)
    has_decode = w.num_seqs > w.num_prefill_seqs
    return {"workload": f"{w.name}: B={w.num_seqs} H={w.num_heads} KVH={w.num_kv_heads} "
                        f"D={w.head_size} bs={w.block_size}",
            "seed": W.SEED_BASE + cfg, "num_blocks": w.num_blocks,
            "l2": "inputs larger than L2 (KV read per step "
                  f"{dec_bytes / 1e9:.2f} GB)" if has_decode else prefill_footprint(w),
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = CFG_OF[args.workload]
    w = W.make_config(cfg)
    cores = host_cores()
    for _ in range(args.warmup):
        pass  # the oracle has no warm state
    vals = []
    sample = None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = oracle_rate(w, budget_s=max(2.0, 20.0 / max(1, args.steps)), threads=cores)
        vals.append(r["value"])
        sample = r["sample"]
        unit = r["unit"]
        threads = r["threads"]
    elapsed = time.perf_counter() - t0
    value = statistics.median(vals)
    one = oracle_rate(w, budget_s=5.0, threads=1)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": elapsed * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, cfg, world),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": sample, "threads": threads,
                             "value_1core": one["value"], "sample_1core": one["sample"]},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return line


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def write_bytes(w: W.Workload) -> int:
    """Bytes kv_cache_write reads and writes: every new token's key and value
    rows in (2-byte elements), the same rows out in the cache's element size."""
    kv_el = 1 if w.kv_cache_dtype == "fp8_e4m3" else 2
    n = int((w.slot_mapping >= 0).sum()) * w.num_kv_heads * w.head_size * 2   # K and V elements
    return n * (2 + kv_el)


def measure(args, cfg: int, world: int, rank: int, local: int, B, full: bool) -> dict:
    """One workload on this GPU: W untimed warm-up steps, then K steps timed
    with CUDA events on the launching stream between barriers (max over
    ranks), each call of the step bracketed by its own events.  ``full``
    adds the end-to-end run through host buffers and the oracle baseline."""
    dev = torch.device("cuda", local)
    w = W.make_config(cfg, scale_down=args.scale_down)
    st = Step(w, dev, B)
    hbm, bf16_burst, bf16_sust, peak_kind = peaks()
    dec_bytes, flops = algorithmic(w)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    B.check_device_error(f"{w.name} warmup")

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        st.run()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_step = max_over_ranks(t_start.elapsed_time(t_end), world) / args.steps
    # The same K steps again with every call bracketed by its own events (the
    # per-call figures).  An event between two calls keeps the second from
    # starting as a programmatic dependent of the first, so the headline pass
    # above has none.
    st.ev.clear()
    for _ in range(args.steps):
        st.run(mark=True)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    write_ms = statistics.mean(a.elapsed_time(b) for a, b, _, _ in st.ev)
    pre_ms = statistics.mean(b.elapsed_time(c) for _, b, c, _ in st.ev)
    dec_ms = statistics.mean(c.elapsed_time(d) for _, _, c, d in st.ev)
    B.check_device_error(f"{w.name} timed region")

    e2e = None
    if full:
        pin = lambda t: t.cpu().pin_memory()
        d_in = [st.query, st.key, st.value, st.slots, st.tables, st.seq_lens]
        h_in = [pin(t) for t in d_in]
        h_out = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
        h2d, d2h = step_io_bytes(st)
        for _ in range(max(1, args.warmup)):
            for h, d in zip(h_in, d_in):
                d.copy_(h, non_blocking=True)
            st.run()
            h_out.copy_(st.out, non_blocking=True)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            for h, d in zip(h_in, d_in):
                d.copy_(h, non_blocking=True)
            st.run()
            h_out.copy_(st.out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
        e2e = {"ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # ---- metric and per-call figures ---------------------------------------
    traffic = (profiled_traffic(*PROFILE_OF[cfg])
               if cfg in PROFILE_OF and args.scale_down == 1 else None)
    decode = prefill = None
    if st.has_decode:
        gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
        decode = {"kernel": ("paged_attn_decode_multi (split pass, + combine when split)"
                             if w.multi_query_len else
                             "paged_attn_decode (split-KV pass, + combine when split)"),
                  "gbs": gbs, "frac_of_hbm": gbs / hbm, "avg_launch_ms": dec_ms,
                  "algorithmic_bytes_per_launch": dec_bytes}
    if st.has_prefill:
        tf = flops / (pre_ms * 1e-3) / 1e12
        prefill = {"kernel": "paged_attn_prefill_varlen", "tflops": tf,
                   "frac_of_bf16_burst": tf / bf16_burst, "frac_of_bf16_sustained": tf / bf16_sust,
                   "avg_launch_ms": pre_ms, "algorithmic_flops_per_launch": flops}
    if st.has_decode:
        units = (w.num_seqs - w.num_prefill_seqs) * max(1, w.multi_query_len) * world
        value, unit = units / (ms_step * 1e-3), "tokens/s"
        e2e_value = units / (e2e["ms_per_step"] * 1e-3) if e2e else None
    else:
        value, unit = flops * world / (ms_step * 1e-3) / 1e12, "TFLOP/s"
        e2e_value = flops * world / (e2e["ms_per_step"] * 1e-3) / 1e12 if e2e else None
    # the roofline object describes the call that takes most of the step; the
    # profiled traffic belongs to it only if the summary is of that kernel
    decode_roof = bool(decode and (not prefill or dec_ms >= pre_ms))
    if traffic is not None and PROFILE_OF[cfg][0].startswith("decode") != decode_roof:
        traffic = None
    if decode_roof:
        roof = {"bound": "hbm", "achieved": decode["gbs"], "peak": hbm, "unit": "GB/s",
                "frac": decode["frac_of_hbm"], "traffic": traffic, "kernel": decode["kernel"],
                "peak_kind": peak_kind, "algorithmic_bytes_per_launch": dec_bytes,
                "avg_launch_ms": dec_ms}
    else:
        roof = {"bound": "tensor", "achieved": prefill["tflops"], "peak": bf16_burst,
                "unit": "TFLOP/s", "frac": prefill["frac_of_bf16_burst"], "traffic": traffic,
                "kernel": prefill["kernel"], "peak_kind": peak_kind,
                "algorithmic_flops_per_launch": flops, "avg_launch_ms": pre_ms,
                "frac_of_sustained": prefill["frac_of_bf16_sustained"]}
    wb = write_bytes(w)
    write = {"tokens": int(w.slot_mapping.numel()), "us": write_ms * 1e3,
             "gbs": wb / (write_ms * 1e-3) / 1e9, "frac_of_hbm": wb / (write_ms * 1e-3) / 1e9 / hbm,
             "algorithmic_bytes_per_launch": wb}

    block_moves = time_block_moves(st, w, B, args, hbm) if w.copy_pairs.numel() else None

    cpu = None
    if full and rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_budget)

    rec = {"value": value, "unit": unit, "ms_per_step": ms_step, "steps": args.steps,
           "warmup": args.warmup, "config": config_of(w, cfg, world), "roofline": roof,
           "kv_cache_write": write, "clocks": clocks,
           "gpu_launches": st.launches_per_step() * args.steps}
    if decode:
        rec["decode"] = decode
    if prefill:
        rec["prefill"] = prefill
    if block_moves:
        rec["block_moves"] = block_moves
    if full:
        rec["e2e"] = {"value": e2e_value, "unit": unit,
                      "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                      "d2h_bytes_per_step": e2e["d2h_bytes_per_step"]}
        rec["cpu_baseline"] = cpu
    rec["dtype"] = "bf16" if w.dtype == torch.bfloat16 else "fp16"
    del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


# Workloads the default run measures beside the headline decode, by name in
# the line's ``workloads`` object.
EXTRA_OF = {"prefill": "varlen_prefill", "mixed": "mixed_chunked_alibi",
            "swa": "swa_long_decode", "encoder": "encoder_varlen_prefill",
            "decode_fp8": "llama3_8b_decode_fp8", "prefill_fp8": "varlen_prefill_fp8",
            "spec_decode": "llama3_8b_spec_decode"}


def extra_workloads(args) -> list:
    if args.extra == "auto":
        return (["prefill", "mixed", "swa"]
                if args.workload == "decode" and args.scale_down == 1 else [])
    if args.extra in ("", "none"):
        return []
    names = [x.strip() for x in args.extra.split(",") if x.strip()]
    for n in names:
        if n not in EXTRA_OF:
            raise SystemExit(f"--extra: unknown workload {n!r} (choose from {sorted(EXTRA_OF)})")
    return names


def run_ours(args, world, rank, local):
    from paged_kv_cache_246_gb300 import binding as B
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = CFG_OF[args.workload]
    head = measure(args, cfg, world, rank, local, B, full=True)
    subs = {}
    for name in extra_workloads(args):
        rec = measure(args, CFG_OF[name], world, rank, local, B, full=False)
        rec.pop("dtype", None)
        subs[EXTRA_OF[name]] = rec
    if rank != 0:
        return None
    line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": head["dtype"], "data": "synthetic", "config": head["config"],
            "roofline": head["roofline"], "clocks": head["clocks"], "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"], "cpu_baseline": head["cpu_baseline"],
            "kv_cache_write": head["kv_cache_write"]}
    for k in ("decode", "prefill", "block_moves"):
        if k in head:
            line[k] = head[k]
    if subs:
        line["workloads"] = subs
    print(json.dumps(line), flush=True)
    return line


def run_dcp_share(args, world, rank, local):
    """One rank's step of a decode spread over a 2-rank decode context
    parallel group, on this GPU: the cache write of the new tokens the rank
    holds, its share over its half of every sequence's tokens, and the merge
    of the two shares.  The peer's share is computed once beforehand and
    stands in for the all-gather, which one GPU cannot time."""
    from paged_kv_cache_246_gb300 import binding as B
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    R, me = 2, 0
    w = W.make_config(2, scale_down=args.scale_down)
    st = Step(w, dev, B)
    B.kv_cache_write(st.key, st.value, st.cache, st.slots, st.p)   # the whole cache, once
    torch.cuda.synchronize()
    shards = W.shard_for_dcp(st.cache.cpu(), w.block_tables, w.seq_lens, w.block_size, R)
    caches = [c.to(dev) for c, _ in shards]
    tables = [t.to(dev) for _, t in shards]
    # the new token of sequence b (position L_b - 1) and its slot on its rank
    mine = [b for b, L in enumerate(w.seq_lens.tolist()) if (L - 1) % R == me]
    bs = w.block_size
    slots = torch.tensor([int(shards[me][1][b, ((L - 1) // R) // bs]) * bs + ((L - 1) // R) % bs
                          for b, L in ((b, int(w.seq_lens[b])) for b in mine)], dtype=torch.int64)
    key_me, val_me = st.key[mine].contiguous(), st.value[mine].contiguous()
    slots_me = slots.to(dev)
    Bn, H, D = w.num_seqs, w.num_heads, w.head_size
    mx = int(w.seq_lens.max())
    ws_bytes = B.paged_attn_decode_dcp_workspace_size(Bn, 1, mx, R, st.p)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    launches = 1 + (2 if ws_bytes > 0 else 1) + 1   # write, share (+ split combine), merge
    parts_o = torch.empty((R, Bn * H, D), dtype=torch.float32, device=dev)
    parts_ml = torch.empty((R, Bn * H, 2), dtype=torch.float32, device=dev)
    for k in range(R):   # the peer's share, as the all-gather would deliver it
        B.paged_attn_decode_dcp_partial(parts_o[k], parts_ml[k], st.query, caches[k], tables[k],
                                        st.seq_lens, 1, mx, R, k, st.p, ws)
    out = torch.empty_like(st.query)
    hbm, _, _, peak_kind = peaks()
    row = w.num_kv_heads * w.head_size
    kv_bytes = sum(((L - me + R - 1) // R) * row * 2 * 2 for L in w.seq_lens.tolist())
    share_bytes = kv_bytes + Bn * H * D * 2 + Bn * H * (D + 2) * 4          # K/V, q in, share out
    merge_bytes = R * Bn * H * (D + 2) * 4 + Bn * H * D * 2                  # shares in, out
    stream = torch.cuda.current_stream()

    def step(ev=None):
        B.kv_cache_write(key_me, val_me, caches[me], slots_me, st.p)
        if ev is not None:
            ev[0].record(stream)
        B.paged_attn_decode_dcp_partial(parts_o[me], parts_ml[me], st.query, caches[me],
                                        tables[me], st.seq_lens, 1, mx, R, me, st.p, ws)
        if ev is not None:
            ev[1].record(stream)
        B.paged_attn_dcp_combine(out, parts_o, parts_ml, st.p)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    B.check_device_error("dcp warmup")
    sampler = ClockSampler(local)
    sampler.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    B.check_device_error("dcp timed region")
    ms_step = t0.elapsed_time(t1) / args.steps
    share_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in evs)
    merge_ms = statistics.mean(b.elapsed_time(c) for _, b, c in evs)
    achieved = share_bytes / (share_ms * 1e-3) / 1e9
    line = {"metric": METRIC, "value": Bn / (ms_step * 1e-3), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"llama3_8b_decode as rank 0 of a 2-rank decode context "
                                   f"parallel group: B={Bn} H={H} KVH={w.num_kv_heads} D={D} "
                                   f"bs={bs} (peer share precomputed: the all-gather is not "
                                   f"timed)", "seed": W.SEED_BASE + 2,
                       "l2": f"inputs larger than L2 (KV read per step {kv_bytes / 1e9:.2f} GB)",
                       "parallelism": "dcp2 rank share on 1 GPU"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": None,
                         "kernel": "paged_attn_decode_dcp_partial (split pass, + combine when split)",
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": share_bytes,
                         "avg_launch_ms": share_ms},
            "merge": {"ms": merge_ms, "gbs": merge_bytes / (merge_ms * 1e-3) / 1e9},
            "clocks": clocks, "e2e": None, "gpu_launches": launches * args.steps,
            "cpu_baseline": None}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(CFG_OF), default="decode")
    ap.add_argument("--extra", default="auto",
                    help="comma list of workloads measured after the headline and reported in "
                         "its line's 'workloads' object (auto: prefill,mixed,swa beside the "
                         "default decode; none: only the headline)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work per timing (all cores, then one core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scale-down", type=int, default=1,
                    help="divide the batch (for small profiling captures only)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.workload == "dcp2_share":
        run_dcp_share(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
