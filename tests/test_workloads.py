"""The seeded input generators (CPU only)."""
import torch

from paged_kv_cache_246_gb300 import workloads as W


def test_deterministic():
    a = W.make_config(1)
    b = W.make_config(1)
    for f in ("seq_lens", "block_tables", "kv_cache", "query", "key", "value",
              "slot_mapping"):
        assert torch.equal(getattr(a, f).view(torch.uint8) if getattr(a, f).is_floating_point() else getattr(a, f),
                           getattr(b, f).view(torch.uint8) if getattr(b, f).is_floating_point() else getattr(b, f))


def test_tiny_decode_recipe():
    w = W.make_config(1)
    assert w.dtype == torch.float16 and w.num_blocks == 32
    assert (w.num_heads, w.num_kv_heads, w.head_size, w.block_size) == (4, 2, 64, 16)
    assert w.seq_lens.min() >= 1 and w.seq_lens.max() <= 100
    assert w.kv_cache.shape == (2, 32, 16 * 2 * 64)


def test_block_tables_are_distinct_blocks():
    w = W.make_config(2, scale_down=16)
    used = []
    for b in range(w.num_seqs):
        n = (int(w.seq_lens[b]) + 15) // 16
        used += w.block_tables[b, :n].tolist()
    assert len(set(used)) == len(used)
    assert max(used) < w.num_blocks
    assert w.num_blocks == -(-len(used) * 11 // 10)


def test_slot_encoding_matches_worked_example():
    # block 2 offset 3 with block size 16 is slot 35 (cpu_attn slot_mapping
    # comment); the generator's scheduler encoding must produce exactly that
    g = torch.Generator().manual_seed(0)
    w = W.build(name="t", g=g, dtype=torch.bfloat16, num_heads=1,
                num_kv_heads=1, head_size=8, block_size=16, seq_lens=[36],
                query_lens=[1], num_prefill_seqs=0, num_blocks=3)
    assert int(w.slot_mapping[0]) == int(w.block_tables[0, 2]) * 16 + 3


def test_cu_from_lengths_worked_example():
    assert W.cu_from_lengths(torch.tensor([4, 6])).tolist() == [0, 4, 10]


def test_mixed_layout_prefill_first():
    w = W.make_config(4, scale_down=8)
    P = w.num_prefill_seqs
    assert P == 1 and (w.query_lens[P:] == 1).all()
    q, cuq, cuk, bt, mq, mk = w.prefill_slices()
    assert q.shape[0] == int(cuq[-1]) and bt.shape[0] == P
    assert (cuk[1:] - cuk[:-1] >= cuq[1:] - cuq[:-1]).all()
    dq, dbt, dsl, dmax = w.decode_slices()
    assert dq.shape[0] == w.num_seqs - P and dmax == int(dsl.max())
    assert w.alibi_slopes is not None and abs(float(w.alibi_slopes[0]) - 2 ** -0.25) < 1e-7


def test_alibi_slopes_standard():
    s = W.alibi_slopes(8)
    assert torch.allclose(s, torch.tensor([2.0 ** -(i) for i in range(1, 9)]))
