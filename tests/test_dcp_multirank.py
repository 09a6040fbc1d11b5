"""Decode context parallelism's exchange step on CPU: two gloo ranks.

Each rank holds the tokens j % 2 == rank of every sequence, computes its
share over them (here with the oracle: the CPU stands in for the GPU's
paged_attn_decode_dcp_partial), and the library's gather_shares all-gathers
the shares rank-major; merged with a3 they must give the decode over whole
sequences on both ranks."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    sys.path.insert(0, ROOT)
    from paged_kv_cache_246_gb300 import workloads as W
    g = torch.Generator().manual_seed(77)
    w = W.build(name="dcp", g=g, dtype=torch.bfloat16, num_heads=4, num_kv_heads=2, head_size=64,
                block_size=16, seq_lens=[3, 40, 91, 130], query_lens=[2, 2, 2, 2],
                num_prefill_seqs=0, alibi=True, sliding_window=50, multi_query_len=2)
    return w


def _params(w):
    import oracle as O
    return O.AttnParams(w.num_heads, w.num_kv_heads, w.head_size, w.block_size, w.scale,
                        w.alibi_slopes.tolist(), w.sliding_window)


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle as O
    from paged_kv_cache_246_gb300 import dcp, workloads as W
    w = _batch()
    p = _params(w)
    cache = w.kv_cache.clone()
    O.kv_cache_write(w.key, w.value, cache, w.slot_mapping, p)
    local_cache, local_tables = W.shard_for_dcp(cache, w.block_tables, w.seq_lens, w.block_size,
                                                world)[rank]
    o, m, l = O.paged_attn_decode_dcp_partials(w.query, local_cache, local_tables, w.seq_lens,
                                               2, world, rank, p)
    H, D = w.num_heads, w.head_size
    part_o = o.view(-1, H, D).reshape(-1, D).float()
    part_ml = torch.stack([m.reshape(-1), l.reshape(-1)], 1).float()
    parts_o, parts_ml = dcp.gather_shares(part_o, part_ml)
    shares = [(parts_o[r].double().view(-1, H * D), parts_ml[r, :, 0].double().view(-1, H),
               parts_ml[r, :, 1].double().view(-1, H)) for r in range(world)]
    merged = O.combine_dcp_partials(shares, H, D)
    torch.save(merged, os.path.join(out_dir, f"r{rank}.pt"))
    dist.destroy_process_group()


def test_two_gloo_ranks_gather_shares_into_the_decode(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    sys.path.insert(0, ROOT)
    import oracle as O
    w = _batch()
    p = _params(w)
    cache = w.kv_cache.clone()
    O.kv_cache_write(w.key, w.value, cache, w.slot_mapping, p)
    ref = O.paged_attn_decode_multi(w.query, cache, w.block_tables, w.seq_lens, 2, p)
    for r in range(world):
        got = torch.load(tmp_path / f"r{r}.pt")
        err = (got - ref).abs().max().item()
        assert err < 1e-5, (r, err)   # shares crossed the exchange in fp32
