"""Seeded synthetic inputs for the paged-KV attention path.

This module only draws inputs: lengths, block placement, the metadata an
engine's scheduler would hand to the attention layer (block tables,
slot_mapping, cu-seqlens), N(0,1) queries/keys/values and cache contents.
It holds none of the attention arithmetic.  Tests, the smoke check and the
bench draw from it, and the same CPU tensors feed both the CUDA library (after
a copy to the device) and the fp64 oracle, so both see identical bits.

The five named workloads follow the attention-backend pages' metadata
(xformers.py XFormersMetadata, cpu_attn TorchSDPAMetadata):

1. ``tiny_decode``: fp16, 4 seqs, 4/2 heads, head 64, block 16, seq_len in
   U[1,100], a 32-block pool, tables a random permutation.
2. ``llama3_8b_decode``: bf16, 256 seqs, 32/8 heads, head 128, block 16,
   seq_len in U[512,4096], pool = needed blocks + 10%.
3. ``varlen_prefill``: bf16, 16 prompts, lengths log-uniform in [128,8192],
   no cached context.
4. ``mixed_chunked_alibi``: bf16, 8 prefill chunks (q in U[256,2048] on a
   cached context in U[0,8192]) followed by 192 decodes (seq_len in
   U[256,8192]); ALiBi slopes 2^(-8i/num_heads), i = 1..num_heads.
5. ``swa_long_decode``: bf16, 64 seqs, seq_len in U[16384,32768], window
   4096, then 2048 block copies and a 4096-block swap out to pinned host
   memory and back.
6. ``encoder_varlen_prefill``: the shape of 3 with non-causal (encoder)
   attention: every query row sees its whole prompt.
7. ``llama3_8b_decode_fp8``: the shape of 2 with an fp8 (E4M3) cache,
   k_scale = v_scale = 0.02 (N(0,1) keys and values map to codes of up to
   about +-250, inside E4M3's +-448).
8. ``varlen_prefill_fp8``: the shape of 3 over an fp8 (E4M3) cache with the
   same scales as 7 (the prompts' keys and values are quantised by the
   cache write).
9. ``llama3_8b_spec_decode``: the shape of 2 with 128 sequences each
   decoding 4 tokens (1 + 3 speculative, a uniform batch).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

SEED_BASE = 1000

__all__ = ["Workload", "build", "CONFIGS", "make_config", "alibi_slopes",
           "cu_from_lengths", "fill_normal", "shard_for_dcp"]


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    scale: float
    alibi_slopes: Optional[torch.Tensor]     # fp32 [num_heads] or None
    sliding_window: int                      # <= 0: none
    seq_lens: torch.Tensor                   # int32 [B]: length after the step
    query_lens: torch.Tensor                 # int32 [B]: new tokens this step
    num_prefill_seqs: int                    # sequences [0, P) are prefill
    block_tables: torch.Tensor               # int32 [B, max_blocks_per_seq]
    kv_cache: torch.Tensor                   # [2, NB, bs*KVH*D], context filled
    query: torch.Tensor                      # [T, H*D]
    key: torch.Tensor                        # [T, KVH*D]
    value: torch.Tensor                      # [T, KVH*D]
    slot_mapping: torch.Tensor               # int64 [T]
    copy_pairs: torch.Tensor = field(default_factory=lambda: torch.empty(0, 2, dtype=torch.int64))
    swap_pairs: torch.Tensor = field(default_factory=lambda: torch.empty(0, 2, dtype=torch.int64))
    causal: bool = True                      # False: encoder attention
    kv_cache_dtype: str = "auto"             # or "fp8_e4m3" (uint8 cache)
    k_scale: float = 1.0
    v_scale: float = 1.0
    multi_query_len: int = 0                 # > 0: a uniform batch of decodes
                                             # of this many tokens each

    # -- views used by the calls --------------------------------------------
    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def num_prefill_tokens(self) -> int:
        return int(self.query_lens[:self.num_prefill_seqs].sum())

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def prefill_slices(self):
        """(query, cu_seqlens_q, cu_seqlens_k, block_tables, max_q, max_k)."""
        P, Tp = self.num_prefill_seqs, self.num_prefill_tokens
        ql = self.query_lens[:P]
        sl = self.seq_lens[:P]
        return (self.query[:Tp], cu_from_lengths(ql), cu_from_lengths(sl),
                self.block_tables[:P],
                int(ql.max()) if P else 0, int(sl.max()) if P else 0)

    def decode_slices(self):
        """(query, block_tables, seq_lens, max_seq_len)."""
        P, Tp = self.num_prefill_seqs, self.num_prefill_tokens
        sl = self.seq_lens[P:]
        return (self.query[Tp:], self.block_tables[P:], sl,
                int(sl.max()) if sl.numel() else 0)


def shard_for_dcp(kv_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                  block_size: int, world: int):
    """Lay a batch's cached tokens out over ``world`` decode context parallel
    ranks: token j of a sequence goes to rank j % world at local position
    j // world (layout only, no attention arithmetic).  Returns per rank
    (local_cache, local_tables), each cache [2, NB_r, row * block_size] with
    the rank's tokens in local order behind a fresh block table."""
    bs = block_size
    row = kv_cache.shape[2] // bs
    B = seq_lens.numel()
    out = []
    for r in range(world):
        lens = [max(0, (int(L) - r + world - 1) // world) for L in seq_lens.tolist()]
        nblk = [(Lr + bs - 1) // bs for Lr in lens]
        NB = max(1, sum(nblk))
        cache = torch.zeros(2, NB, bs * row, dtype=kv_cache.dtype)
        tables = torch.zeros(B, max(1, max(nblk) if nblk else 1), dtype=torch.int32)
        k = 0
        for b in range(B):
            for lb in range(nblk[b]):
                tables[b, lb] = k
                k += 1
            for jl in range(lens[b]):
                j = jl * world + r
                src_blk, src_off = int(block_tables[b, j // bs]), j % bs
                dst_blk, dst_off = int(tables[b, jl // bs]), jl % bs
                cache[:, dst_blk, dst_off * row:(dst_off + 1) * row] = \
                    kv_cache[:, src_blk, src_off * row:(src_off + 1) * row]
        out.append((cache, tables))
    return out


def cu_from_lengths(lengths: torch.Tensor) -> torch.Tensor:
    """[l0, l1, ...] -> int32 [0, l0, l0+l1, ...] (batch+1 entries)."""
    out = torch.zeros(lengths.numel() + 1, dtype=torch.int32)
    out[1:] = torch.cumsum(lengths.to(torch.int64), 0).to(torch.int32)
    return out


def alibi_slopes(num_heads: int) -> torch.Tensor:
    """Standard geometric ALiBi slopes 2^(-8 i / num_heads), i = 1..num_heads."""
    return torch.tensor([2.0 ** (-8.0 * i / num_heads)
                         for i in range(1, num_heads + 1)], dtype=torch.float32)


def fill_normal(n: int, dtype: torch.dtype, g: torch.Generator,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """n N(0,1) samples rounded to ``dtype``, drawn in fp32 in chunks."""
    if out is None:
        out = torch.empty(n, dtype=dtype)
    chunk = 1 << 26
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        out[a:b] = torch.randn(b - a, generator=g, dtype=torch.float32)
    return out


def _uniform_int(g, n, lo, hi) -> torch.Tensor:
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64)


def _log_uniform_int(g, n, lo, hi) -> torch.Tensor:
    u = torch.rand(n, generator=g, dtype=torch.float64)
    x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return torch.round(x).to(torch.int64).clamp(lo, hi)


def build(*, name: str, g: torch.Generator, dtype: torch.dtype,
          num_heads: int, num_kv_heads: int, head_size: int, block_size: int,
          seq_lens, query_lens, num_prefill_seqs: int,
          num_blocks: Optional[int] = None, pool_extra: float = 0.10,
          alibi: bool = False, sliding_window: int = 0,
          n_copy: int = 0, n_swap: int = 0, fill_cache: bool = True,
          causal: bool = True, kv_cache_dtype: str = "auto", k_scale: float = 1.0,
          v_scale: float = 1.0, multi_query_len: int = 0) -> Workload:
    """Lay out a batch in a paged pool and draw its tensors.

    Block placement: the N = sum ceil(seq_len / block_size) blocks the batch
    needs are the first N entries of a random permutation of the pool's
    blocks, dealt to the sequences' logical blocks in order; the rest of the
    pool is free.  Every slot of the pool is filled with N(0,1) (so all cached
    context exists); the step's new tokens get fresh N(0,1) K/V and their
    slots (the last query_len positions of each sequence) in slot_mapping.
    """
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int64)
    query_lens = torch.as_tensor(query_lens, dtype=torch.int64)
    B = seq_lens.numel()
    if multi_query_len:  # every sequence decodes multi_query_len tokens
        assert num_prefill_seqs == 0 and bool((query_lens == multi_query_len).all())
    assert bool((query_lens <= seq_lens).all()) and bool((query_lens >= 0).all())
    bs = block_size
    nblk = [(int(L) + bs - 1) // bs for L in seq_lens]
    need = sum(nblk)
    if num_blocks is None:
        permille = round(pool_extra * 1000)
        num_blocks = max(1, need + -(-need * permille // 1000))
    assert need <= num_blocks, "pool too small for the batch"
    perm = torch.randperm(num_blocks, generator=g)
    maxblk = max(1, max(nblk) if nblk else 1)
    tables = torch.zeros(B, maxblk, dtype=torch.int32)
    used = []
    k = 0
    for b in range(B):
        for lb in range(nblk[b]):
            tables[b, lb] = int(perm[k])
            used.append(int(perm[k]))
            k += 1
    free = [int(x) for x in perm[need:]]

    row = num_kv_heads * head_size
    if kv_cache_dtype == "fp8_e4m3":
        # cached context as 8-bit codes: N(0,1) / scale narrowed by torch's
        # float8_e4m3fn conversion (input drawing only; values stay in range)
        kv_cache = torch.zeros(2, num_blocks, bs * row, dtype=torch.uint8)
        if fill_cache:
            for half, sc in ((0, k_scale), (1, v_scale)):
                flat = kv_cache[half].view(-1)
                for a in range(0, flat.numel(), 1 << 26):
                    b = min(flat.numel(), a + (1 << 26))
                    x = torch.randn(b - a, generator=g, dtype=torch.float32) / sc
                    flat[a:b] = x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    else:
        kv_cache = torch.zeros(2, num_blocks, bs * row, dtype=dtype)
        if fill_cache:
            fill_normal(kv_cache.numel(), dtype, g, out=kv_cache.view(-1))

    T = int(query_lens.sum())
    query = fill_normal(T * num_heads * head_size, dtype, g).view(T, -1)
    key = fill_normal(T * row, dtype, g).view(T, row)
    value = fill_normal(T * row, dtype, g).view(T, row)

    # The scheduler's slot assignment for the new tokens: the last query_len
    # positions of each sequence, at (table[pos // bs], pos % bs).
    slots = torch.empty(T, dtype=torch.int64)
    t = 0
    for b in range(B):
        L, q = int(seq_lens[b]), int(query_lens[b])
        for pos in range(L - q, L):
            slots[t] = int(tables[b, pos // bs]) * bs + pos % bs
            t += 1

    copy_pairs = torch.empty(0, 2, dtype=torch.int64)
    if n_copy:
        assert n_copy <= len(free)
        src_idx = torch.randint(0, len(used), (n_copy,), generator=g)
        dst_idx = torch.randperm(len(free), generator=g)[:n_copy]
        copy_pairs = torch.tensor([[used[int(a)], free[int(d)]]
                                   for a, d in zip(src_idx, dst_idx)],
                                  dtype=torch.int64).view(-1, 2)
    swap_pairs = torch.empty(0, 2, dtype=torch.int64)
    if n_swap:
        # swap-out list: distinct used device blocks -> host blocks 0..n-1
        assert n_swap <= len(used)
        pick = torch.randperm(len(used), generator=g)[:n_swap]
        swap_pairs = torch.tensor([[used[int(a)], k] for k, a in enumerate(pick)],
                                  dtype=torch.int64).view(-1, 2)

    return Workload(
        name=name, dtype=dtype, num_heads=num_heads,
        num_kv_heads=num_kv_heads, head_size=head_size, block_size=bs,
        num_blocks=num_blocks, scale=1.0 / math.sqrt(head_size),
        alibi_slopes=alibi_slopes(num_heads) if alibi else None,
        sliding_window=sliding_window,
        seq_lens=seq_lens.to(torch.int32), query_lens=query_lens.to(torch.int32),
        num_prefill_seqs=num_prefill_seqs, block_tables=tables,
        kv_cache=kv_cache, query=query, key=key, value=value,
        slot_mapping=slots, copy_pairs=copy_pairs, swap_pairs=swap_pairs,
        causal=causal, kv_cache_dtype=kv_cache_dtype, k_scale=k_scale, v_scale=v_scale,
        multi_query_len=multi_query_len)


# ---------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------

def _tiny_decode(g, scale_down=1):
    B = 4
    L = _uniform_int(g, B, 1, 100)
    return build(name="tiny_decode", g=g, dtype=torch.float16, num_heads=4,
                 num_kv_heads=2, head_size=64, block_size=16, seq_lens=L,
                 query_lens=torch.ones(B, dtype=torch.int64),
                 num_prefill_seqs=0, num_blocks=32)


def _llama3_8b_decode(g, scale_down=1):
    B = max(1, 256 // scale_down)
    L = _uniform_int(g, B, 512, 4096)
    return build(name="llama3_8b_decode", g=g, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                 seq_lens=L, query_lens=torch.ones(B, dtype=torch.int64),
                 num_prefill_seqs=0)


def _varlen_prefill(g, scale_down=1):
    B = max(1, 16 // scale_down)
    L = _log_uniform_int(g, B, 128, 8192)
    return build(name="varlen_prefill", g=g, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                 seq_lens=L, query_lens=L, num_prefill_seqs=B)


def _mixed_chunked_alibi(g, scale_down=1):
    P = max(1, 8 // scale_down)
    Dn = max(1, 192 // scale_down)
    q = _uniform_int(g, P, 256, 2048)
    c = _uniform_int(g, P, 0, 8192)
    Ld = _uniform_int(g, Dn, 256, 8192)
    seq_lens = torch.cat([q + c, Ld])
    query_lens = torch.cat([q, torch.ones(Dn, dtype=torch.int64)])
    return build(name="mixed_chunked_alibi", g=g, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                 seq_lens=seq_lens, query_lens=query_lens, num_prefill_seqs=P,
                 alibi=True)


def _swa_long_decode(g, scale_down=1):
    B = max(1, 64 // scale_down)
    L = _uniform_int(g, B, 16384, 32768)
    return build(name="swa_long_decode", g=g, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                 seq_lens=L, query_lens=torch.ones(B, dtype=torch.int64),
                 num_prefill_seqs=0, sliding_window=4096,
                 n_copy=max(1, 2048 // scale_down),
                 n_swap=max(1, 4096 // scale_down))


def _encoder_varlen_prefill(g, scale_down=1):
    B = max(1, 16 // scale_down)
    L = _log_uniform_int(g, B, 128, 8192)
    return build(name="encoder_varlen_prefill", g=g, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                 seq_lens=L, query_lens=L, num_prefill_seqs=B, causal=False)


def _varlen_prefill_fp8(g, scale_down=1):
    B = max(1, 16 // scale_down)
    L = _log_uniform_int(g, B, 128, 8192)
    return build(name="varlen_prefill_fp8", g=g, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                 seq_lens=L, query_lens=L, num_prefill_seqs=B, kv_cache_dtype="fp8_e4m3",
                 k_scale=0.02, v_scale=0.02)


def _llama3_8b_spec_decode(g, scale_down=1):
    B = max(1, 128 // scale_down)
    q = 4  # one token + 3 speculative tokens per sequence
    L = _uniform_int(g, B, 512, 4096)
    return build(name="llama3_8b_spec_decode", g=g, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                 seq_lens=L, query_lens=torch.full((B,), q, dtype=torch.int64),
                 num_prefill_seqs=0, multi_query_len=q)


def _llama3_8b_decode_fp8(g, scale_down=1):
    B = max(1, 256 // scale_down)
    L = _uniform_int(g, B, 512, 4096)
    return build(name="llama3_8b_decode_fp8", g=g, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                 seq_lens=L, query_lens=torch.ones(B, dtype=torch.int64),
                 num_prefill_seqs=0, kv_cache_dtype="fp8_e4m3", k_scale=0.02,
                 v_scale=0.02)


CONFIGS = {
    1: _tiny_decode,
    2: _llama3_8b_decode,
    3: _varlen_prefill,
    4: _mixed_chunked_alibi,
    5: _swa_long_decode,
    6: _encoder_varlen_prefill,
    7: _llama3_8b_decode_fp8,
    8: _varlen_prefill_fp8,
    9: _llama3_8b_spec_decode,
}


def make_config(index: int, scale_down: int = 1) -> Workload:
    """Workload ``index`` (1..9) drawn from generator seed 1000 + index.

    ``scale_down`` > 1 divides the batch counts (not the lengths), for tests
    that want the shape of a workload at a fraction of its size.
    """
    g = torch.Generator().manual_seed(SEED_BASE + index)
    return CONFIGS[index](g, scale_down)
