"""Plain fp64 CPU restatement of attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg; never by the library.  It shares no code
with the CUDA path.  Every function is the plain definition of what one step of
the hot path computes, written for a reader to check against the source pages
by eye.  Plain torch CPU ops are used, floating point in fp64; the inputs are
the same fp16/bf16 bits the GPU sees, widened exactly.

Sources (cited by page title and the class, function or comment on it):

* "aphrodite-engine/aphrodite/attention/backends/xformers.py" (written
  ``xformers.py`` below): ``XFormersBackend``, ``XFormersMetadata`` (the
  context_len / subquery_len / seqlen diagram and the cu-seqlens example),
  ``XFormersImpl.forward``, ``_run_memory_efficient_xformers_forward``,
  ``_make_alibi_bias``.
* "vllm.v1.attention.backends.cpu_attn" (``cpu_attn`` below):
  ``TorchSDPABackendImpl.forward``, ``_run_sdpa_forward``,
  ``TorchSDPAMetadata`` (the slot_mapping and block_tables comments).
* "vllm.v1.attention.backends.utils" (``backends.utils`` below):
  ``CommonAttentionMetadata`` (query_start_loc, seq_lens,
  num_computed_tokens).

Readings taken where the pages are silent:

* cache block layout: the pages print only the flat size
  ``block_size * num_kv_heads * head_size`` of one block.  Read token-major,
  ``[block_size][num_kv_heads][head_size]``, so a cache slot holds one key
  (or value) row exactly as it appears in ``key[t]``.
* sliding window W > 0: a query at position i sees keys ``i - W < j <= i``
  (exactly W keys including itself); W <= 0 means no window.
* ALiBi together with a window: both apply (the pages drop the window when
  ALiBi is set; ``drop_window_with_alibi=True`` reproduces that instead).
* a sequence with no keys (decode ``seq_len == 0``) outputs zeros.
* a negative slot in ``slot_mapping`` is a padding token: nothing is written.
"""
from __future__ import annotations

import bisect
import math
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

F64 = torch.float64

__all__ = [
    "AttnParams", "slot_location", "cache_row", "kv_cache_write",
    "kv_head_of", "window_lo", "alibi_bias", "decode_position",
    "lengths_from_cu", "gather_kv", "attend_rows", "paged_attn_decode",
    "paged_attn_prefill_varlen", "decode_split_partials",
    "combine_split_partials", "kv_copy_blocks", "kv_swap_blocks",
    "e4m3_decode", "e4m3_encode", "fp8_quantize", "multi_decode_position",
    "paged_attn_decode_multi", "dcp_local_seq_len", "dcp_global_position",
    "paged_attn_decode_dcp_partials", "combine_dcp_partials",
]


@dataclass(frozen=True)
class AttnParams:
    """Per-layer attention constants.

    Mirrors the constructor arguments of ``XFormersImpl`` (xformers.py) and
    ``TorchSDPABackendImpl`` (cpu_attn): num_heads, head_size, scale,
    num_kv_heads, alibi_slopes, sliding_window; plus the cache block size and
    ``causal`` (cpu_attn ``_run_sdpa_forward`` is causal only for decoder
    attention; encoder and encoder-only attention see the whole sequence).
    """
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    scale: float
    alibi_slopes: Optional[Sequence[float]] = None
    sliding_window: int = 0
    causal: bool = True
    kv_cache_dtype: str = "auto"   # "auto" (model dtype) or "fp8_e4m3"
    k_scale: float = 1.0           # fp8 cache: key = code * k_scale
    v_scale: float = 1.0           #            value = code * v_scale

    @property
    def queries_per_kv(self) -> int:
        # xformers.py XFormersImpl.__init__: num_heads must be a multiple of
        # num_kv_heads; the ratio is num_queries_per_kv.
        assert self.num_heads % self.num_kv_heads == 0
        return self.num_heads // self.num_kv_heads

    @property
    def row_elems(self) -> int:
        return self.num_kv_heads * self.head_size


# ---------------------------------------------------------------------------
# fp8 cache codes (the kv_cache_dtype / k_scale / v_scale of xformers.py
# write_to_paged_cache and cpu_attn forward_decode).  Reading taken: the
# 8-bit format is E4M3 in its "fn" form (sign, 4 exponent bits with bias 7,
# 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448);
# a value is stored as the code nearest to x / scale (ties to the even
# code), saturating at +-448, with x / scale taken in fp32.
# ---------------------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    """Value of an E4M3 code, from its bit fields."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)   # subnormal
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_POS = [e4m3_decode(c) for c in range(0x7F)]   # codes 0x00..0x7E, increasing


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code to x, ties to the even code, saturating at +-448."""
    if x != x:
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0x00
    a = abs(x)
    if a >= _E4M3_POS[-1]:
        return sign | 0x7E                        # saturate at 448
    hi = bisect.bisect_left(_E4M3_POS, a)        # first code with value >= a
    if _E4M3_POS[hi] == a:
        return sign | hi
    lo = hi - 1                                  # value(lo) < a < value(hi)
    d_lo, d_hi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    if d_lo < d_hi or (d_lo == d_hi and lo % 2 == 0):
        return sign | lo
    return sign | hi


def fp8_quantize(x: torch.Tensor, scale: float) -> torch.Tensor:
    """uint8 codes of x / scale (quotient in fp32, then nearest code)."""
    q = (x.to(torch.float32) / torch.tensor(scale, dtype=torch.float32)).reshape(-1)
    return torch.tensor([e4m3_encode(float(v)) for v in q.tolist()],
                        dtype=torch.uint8).view(x.shape)


_E4M3_TABLE = torch.tensor([e4m3_decode(c) for c in range(256)], dtype=F64)


def _dequant(codes: torch.Tensor, scale: float) -> torch.Tensor:
    return _E4M3_TABLE[codes.to(torch.int64)] * scale


# ---------------------------------------------------------------------------
# a1: the cache write (reshape_and_cache)
# ---------------------------------------------------------------------------

def slot_location(slot: int, block_size: int) -> tuple[int, int]:
    """Slot -> (physical block, offset in block).

    cpu_attn, TorchSDPAMetadata.slot_mapping comment: a slot number names the
    block ``slot // block_size`` and the position ``slot % block_size`` in it
    (its worked example maps slots 35, 2, 17 with block size 16 to block 2,
    block 0 and block 1).
    """
    return slot // block_size, slot % block_size


def cache_row(kv_cache: torch.Tensor, half: int, block: int, offset: int,
              p: AttnParams) -> torch.Tensor:
    """View of one token's row (num_kv_heads * head_size elements).

    Cache shape is ``[2, num_blocks, block_size * num_kv_heads * head_size]``
    (xformers.py XFormersImpl.forward docstring; cpu_attn forward docstring);
    half 0 holds keys, half 1 values.  Token-major reading of a block.
    """
    n = p.row_elems
    return kv_cache[half, block, offset * n:(offset + 1) * n]


def kv_cache_write(key: torch.Tensor, value: torch.Tensor,
                   kv_cache: torch.Tensor, slot_mapping: torch.Tensor,
                   p: AttnParams) -> None:
    """Store each new token's key and value row in its slot, in place.

    xformers.py XFormersImpl.forward / cpu_attn TorchSDPABackendImpl.forward:
    the new key and value are written into the paged cache through
    slot_mapping before any attention runs.  The copy is bitwise (done on
    16-bit integer views).  Negative slots are padding and are skipped.
    With an fp8 cache (uint8 tensor) the row is stored as E4M3 codes of
    key / k_scale and value / v_scale.
    """
    if p.kv_cache_dtype == "fp8_e4m3":
        for t in range(key.shape[0]):
            s = int(slot_mapping[t])
            if s < 0:
                continue
            blk, off = slot_location(s, p.block_size)
            cache_row(kv_cache, 0, blk, off, p).copy_(fp8_quantize(key[t].reshape(-1), p.k_scale))
            cache_row(kv_cache, 1, blk, off, p).copy_(fp8_quantize(value[t].reshape(-1), p.v_scale))
        return
    kc = kv_cache.view(torch.int16)
    kb = key.reshape(key.shape[0], -1).view(torch.int16)
    vb = value.reshape(value.shape[0], -1).view(torch.int16)
    for t in range(key.shape[0]):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        blk, off = slot_location(s, p.block_size)
        cache_row(kc, 0, blk, off, p).copy_(kb[t])
        cache_row(kc, 1, blk, off, p).copy_(vb[t])


# ---------------------------------------------------------------------------
# Small definitions shared by decode and prefill
# ---------------------------------------------------------------------------

def kv_head_of(h: int, queries_per_kv: int) -> int:
    """Query head h reads KV head h // num_queries_per_kv.

    xformers.py _run_memory_efficient_xformers_forward views the query as
    [tokens, num_kv_heads, num_queries_per_kv, head_size]; cpu_attn
    _run_sdpa_forward repeat_interleaves K/V num_queries_per_kv times along
    the head axis.  Both give this mapping.
    """
    return h // queries_per_kv


def window_lo(i: int, window: int) -> int:
    """First key position visible from query position i.

    Causal attention sees keys 0..i; a sliding window W > 0 keeps the W most
    recent of them, i - W < j <= i.
    """
    if window > 0:
        return max(0, i - window + 1)
    return 0


def alibi_bias(slope: float, j, i):
    """ALiBi term added to the score of key j for query position i.

    xformers.py _make_alibi_bias builds ``bias[i][j] = j - i`` (the comment
    there notes the per-row-constant variant ``j`` gives the same softmax) and
    multiplies it by the head's slope.
    """
    return slope * (j - i)


def decode_position(seq_len: int) -> int:
    """Position of the one query token of a decoding sequence.

    xformers.py XFormersMetadata comment: for decoding, context_len already
    counts the new token (it was written to the cache first), so the query
    sits at the last position, seq_len - 1.
    """
    return seq_len - 1


def lengths_from_cu(cu: torch.Tensor) -> list[int]:
    """Per-sequence lengths from a cumulative start-location vector.

    xformers.py XFormersMetadata: subquery_start_loc / seq_start_loc have
    batch+1 entries, e.g. lengths [4, 6] give [0, 4, 10].
    """
    c = [int(x) for x in cu]
    return [c[k + 1] - c[k] for k in range(len(c) - 1)]


def gather_kv(kv_cache: torch.Tensor, table_row: torch.Tensor, n_tokens: int,
              p: AttnParams) -> tuple[torch.Tensor, torch.Tensor]:
    """Logical K/V of one sequence, positions 0..n_tokens-1, as fp64.

    cpu_attn TorchSDPAMetadata.block_tables comment: row b lists the physical
    blocks of sequence b in order; logical position j lives in block
    ``table[j // block_size]`` at offset ``j % block_size``.
    Returns K, V of shape [n_tokens, num_kv_heads, head_size].
    """
    bs = p.block_size
    K = torch.empty(n_tokens, p.num_kv_heads, p.head_size, dtype=F64)
    V = torch.empty_like(K)
    for k in range((n_tokens + bs - 1) // bs):   # logical block k
        blk = int(table_row[k])
        j0, j1 = k * bs, min((k + 1) * bs, n_tokens)
        for half, dst in ((0, K), (1, V)):
            rows = kv_cache[half, blk].view(bs, p.num_kv_heads, p.head_size)[:j1 - j0]
            if p.kv_cache_dtype == "fp8_e4m3":   # code * scale
                dst[j0:j1] = _dequant(rows, p.k_scale if half == 0 else p.v_scale)
            else:
                dst[j0:j1] = rows.to(F64)
    return K, V


def attend_rows(q: torch.Tensor, positions: Sequence[int], K: torch.Tensor,
                V: torch.Tensor, scale: float, slope: Optional[float],
                window: int, causal: bool = True) -> torch.Tensor:
    """softmax(scale * q K^T + alibi + mask) V for a set of query rows.

    q: [n, D] fp64; positions: query position i of each row; K, V: [L, D]
    fp64 holding positions 0..L-1 of one KV head.  Row r sees keys
    ``window_lo(i) <= j <= i`` (causal; xformers.py BlockDiagonalCausalMask,
    cpu_attn is_causal SDPA), scores ``scale * q.k_j`` (plus
    ``alibi_bias``), then a softmax and the weighted sum of V.  With
    ``causal=False`` (encoder attention, cpu_attn ``_run_sdpa_forward``) every
    row sees all keys 0..L-1; a window is not defined there.
    """
    n = q.shape[0]
    out = torch.zeros(n, V.shape[1], dtype=F64)
    for r in range(n):
        i = int(positions[r])
        if causal:
            lo, hi = window_lo(i, window), i
        else:
            assert window <= 0, "a sliding window is only defined for causal attention"
            lo, hi = 0, K.shape[0] - 1
        if hi < lo:
            continue  # no key visible: zeros
        j = torch.arange(lo, hi + 1, dtype=F64)
        s = scale * (K[lo:hi + 1] @ q[r])
        if slope is not None:
            s = s + alibi_bias(slope, j, i)
        e = torch.exp(s - s.max())
        out[r] = (e / e.sum()) @ V[lo:hi + 1]
    return out


def _slope(p: AttnParams, h: int) -> Optional[float]:
    return None if p.alibi_slopes is None else float(p.alibi_slopes[h])


def _window(p: AttnParams, drop_window_with_alibi: bool) -> int:
    if drop_window_with_alibi and p.alibi_slopes is not None:
        return 0
    return p.sliding_window


# ---------------------------------------------------------------------------
# a2 + a3: decode
# ---------------------------------------------------------------------------

def paged_attn_decode(query: torch.Tensor, kv_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor,
                      p: AttnParams, seqs: Optional[Sequence[int]] = None,
                      drop_window_with_alibi: bool = False) -> torch.Tensor:
    """One query token per sequence, K/V gathered through block_tables.

    xformers.py XFormersImpl.forward -> PagedAttention.forward_decode and
    cpu_attn TorchSDPABackendImpl.forward -> forward_decode: query
    [num_seqs, num_heads * head_size], block_tables, seq_lens (including the
    token just written), num_kv_heads, scale, alibi_slopes.
    Returns fp64 [num_seqs, num_heads * head_size]; rows not in ``seqs`` (if
    given) are left NaN.
    """
    B = query.shape[0]
    H, D, qpk = p.num_heads, p.head_size, p.queries_per_kv
    out = torch.full((B, H * D), float("nan"), dtype=F64)
    q_all = query.to(F64).view(B, H, D)
    window = _window(p, drop_window_with_alibi)
    for b in (range(B) if seqs is None else seqs):
        L = int(seq_lens[b])
        if L == 0:
            out[b] = 0.0
            continue
        K, V = gather_kv(kv_cache, block_tables[b], L, p)
        i = decode_position(L)
        for h in range(H):
            g = kv_head_of(h, qpk)
            o = attend_rows(q_all[b, h:h + 1], [i], K[:, g], V[:, g],
                            p.scale, _slope(p, h), window)
            out[b, h * D:(h + 1) * D] = o[0]
    return out


def multi_decode_position(seq_len: int, query_len: int, t: int) -> int:
    """Position of query token t (0-based) of a decode of query_len tokens.

    A decode with speculative tokens appends query_len = 1 + k tokens; the
    sequence length seq_len counts them all (as for a single-token decode,
    xformers.py ``XFormersMetadata`` context_len note), so they are the last
    query_len positions: seq_len - query_len + t.
    """
    return seq_len - query_len + t


def paged_attn_decode_multi(query: torch.Tensor, kv_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor,
                            query_len: int, p: AttnParams,
                            seqs: Optional[Sequence[int]] = None) -> torch.Tensor:
    """A uniform batch of decodes of query_len tokens each (speculative).

    backends.utils ``AttentionCGSupport.UNIFORM_BATCH``: every decode in the
    batch has the same query length, 1 + num_speculative_tokens
    (``AttentionMetadataBuilder._init_reorder_batch_threshold`` pulls such
    decodes to the front for spec-as-decode kernels).  query is
    [num_seqs * query_len, num_heads * head_size], sequence b's tokens at rows
    b * query_len + t; token t sits at ``multi_decode_position`` and attends
    causally (and within the window) to the keys read through block_tables.
    A sequence with seq_len 0 (padding) gives zero rows.  Returns fp64
    [num_seqs * query_len, num_heads * head_size]; sequences not in ``seqs``
    (if given) are left NaN.
    """
    B = seq_lens.numel()
    H, D, qpk = p.num_heads, p.head_size, p.queries_per_kv
    q_all = query.to(F64).view(B, query_len, H, D)
    out = torch.full((B * query_len, H * D), float("nan"), dtype=F64)
    window = _window(p, False)
    for b in (range(B) if seqs is None else seqs):
        L = int(seq_lens[b])
        rows = slice(b * query_len, (b + 1) * query_len)
        if L == 0:
            out[rows] = 0.0
            continue
        assert L >= query_len, "a decode cannot hold more tokens than its sequence"
        K, V = gather_kv(kv_cache, block_tables[b], L, p)
        pos = [multi_decode_position(L, query_len, t) for t in range(query_len)]
        for h in range(H):
            g = kv_head_of(h, qpk)
            o = attend_rows(q_all[b, :, h], pos, K[:, g], V[:, g], p.scale,
                            _slope(p, h), window)
            out[rows, h * D:(h + 1) * D] = o
    return out


def decode_split_partials(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                          i: int, scale: float, slope: Optional[float],
                          window: int, split_tokens: int):
    """Flash-decoding partials for one (sequence, head): a3's inputs.

    The visible keys window_lo(i)..i are cut into consecutive pieces of
    ``split_tokens`` positions; each piece gives (o_s, m_s, l_s): its own
    softmax-normalised output, its score maximum and its sum of
    exp(score - m_s).  Method choice of this library (the pages name
    decode context parallelism, backends.utils CommonAttentionMetadata
    dcp_local_seq_lens, but print no combine).
    """
    lo = window_lo(i, window)
    parts = []
    for a in range(lo, i + 1, split_tokens):
        b = min(a + split_tokens, i + 1)
        j = torch.arange(a, b, dtype=F64)
        s = scale * (K[a:b] @ q)
        if slope is not None:
            s = s + alibi_bias(slope, j, i)
        m = s.max()
        e = torch.exp(s - m)
        parts.append(((e / e.sum()) @ V[a:b], float(m), float(e.sum())))
    return parts


def combine_split_partials(parts) -> torch.Tensor:
    """a3: merge split partials into the full softmax-weighted output.

    o = sum_s exp(m_s - m) l_s o_s / sum_s exp(m_s - m) l_s, m = max_s m_s.
    """
    m = max(ms for _, ms, _ in parts)
    w = [math.exp(ms - m) * ls for _, ms, ls in parts]
    num = sum(wk * o for wk, (o, _, _) in zip(w, parts))
    return num / sum(w)


# ---------------------------------------------------------------------------
# f4: decode context parallelism
# ---------------------------------------------------------------------------

def dcp_local_seq_len(seq_len: int, world: int, rank: int) -> int:
    """Tokens of a sequence of seq_len that rank ``rank`` of a decode
    context parallel group of ``world`` ranks holds (backends.utils
    CommonAttentionMetadata dcp_local_seq_lens).

    The pages give only these local lengths; the reading taken here places
    token j on rank j % world at local position j // world, which keeps the
    ranks' lengths within one of each other.
    """
    return max(0, (seq_len - rank + world - 1) // world)


def dcp_global_position(local_index: int, world: int, rank: int) -> int:
    """Position in the sequence of the rank's local token local_index."""
    return local_index * world + rank


def paged_attn_decode_dcp_partials(query: torch.Tensor, local_cache: torch.Tensor,
                                   local_tables: torch.Tensor, seq_lens: torch.Tensor,
                                   query_len: int, world: int, rank: int,
                                   p: AttnParams):
    """One rank's share of a decode under decode context parallelism.

    The query tokens (query_len per sequence, rows b * query_len + t, at
    positions seq_len - query_len + t) attend to the keys this rank holds,
    read through its own cache and block table (its local tokens in local
    order); the result is the (o, m, l) of a3 over those keys: o the
    softmax-normalised output, m the score maximum, l the sum of
    exp(score - m).  A row with no visible key on this rank gets o = 0,
    m = -inf, l = 0.  Returns fp64 o [rows, heads * head_size], m and l
    [rows, heads].
    """
    B = seq_lens.numel()
    H, D, qpk = p.num_heads, p.head_size, p.queries_per_kv
    q_all = query.to(F64).view(B, query_len, H, D)
    o = torch.zeros(B * query_len, H * D, dtype=F64)
    m = torch.full((B * query_len, H), -math.inf, dtype=F64)
    l = torch.zeros(B * query_len, H, dtype=F64)
    window = _window(p, False)
    for b in range(B):
        L = int(seq_lens[b])
        Lr = dcp_local_seq_len(L, world, rank)
        if L == 0 or Lr == 0:
            continue
        K, V = gather_kv(local_cache, local_tables[b], Lr, p)
        pos = torch.tensor([dcp_global_position(k, world, rank) for k in range(Lr)], dtype=F64)
        for t in range(query_len):
            i = multi_decode_position(L, query_len, t)
            keep = (pos <= i) & (pos >= window_lo(i, window))
            if not bool(keep.any()):
                continue
            r = b * query_len + t
            for h in range(H):
                g = kv_head_of(h, qpk)
                s = p.scale * (K[keep, g] @ q_all[b, t, h])
                sl = _slope(p, h)
                if sl is not None:
                    s = s + alibi_bias(sl, pos[keep], i)
                mm = s.max()
                e = torch.exp(s - mm)
                o[r, h * D:(h + 1) * D] = (e / e.sum()) @ V[keep, g]
                m[r, h] = float(mm)
                l[r, h] = float(e.sum())
    return o, m, l


def combine_dcp_partials(parts, num_heads: int, head_size: int) -> torch.Tensor:
    """Merge every rank's (o, m, l) with a3 (combine_split_partials), row by
    row and head by head; ranks with no visible key (l = 0) drop out."""
    o0 = parts[0][0]
    out = torch.zeros_like(o0)
    D = head_size
    for r in range(o0.shape[0]):
        for h in range(num_heads):
            sel = [(o[r, h * D:(h + 1) * D], float(m[r, h]), float(l[r, h]))
                   for o, m, l in parts if float(l[r, h]) > 0.0]
            if sel:
                out[r, h * D:(h + 1) * D] = combine_split_partials(sel)
    return out


# ---------------------------------------------------------------------------
# a4: varlen causal prefill, with or without a cached context
# ---------------------------------------------------------------------------

def paged_attn_prefill_varlen(query: torch.Tensor, cu_seqlens_q: torch.Tensor,
                              cu_seqlens_k: torch.Tensor,
                              kv_cache: torch.Tensor,
                              block_tables: torch.Tensor, p: AttnParams,
                              rows: Optional[Sequence[int]] = None,
                              drop_window_with_alibi: bool = False
                              ) -> torch.Tensor:
    """Packed prompts (or prompt chunks) attending causally through the cache.

    Per sequence b: q_b = query rows in [cu_q[b], cu_q[b+1]) (subquery_len),
    L_b = cu_k[b+1] - cu_k[b] (seqlen), context c_b = L_b - q_b
    (xformers.py XFormersMetadata diagram; backends.utils
    CommonAttentionMetadata num_computed_tokens = seq_lens - query lens).
    Row t of sequence b sits at position i = c_b + t and attends to keys
    window_lo(i)..i, all read through the block table (the chunk's own K/V
    were stored by the cache write first: xformers.py forward writes before
    forward_prefix).  With c_b = 0 this is the block-diagonal causal prefill
    of _run_memory_efficient_xformers_forward and the per-sequence causal SDPA
    of cpu_attn _run_sdpa_forward.
    With ``p.causal`` False (encoder / encoder-only attention, cpu_attn
    ``_run_sdpa_forward`` with is_causal off) row t sees all L_b keys.
    Returns fp64 [num_query_tokens, num_heads * head_size]; rows not listed in
    ``rows`` (if given) are left NaN.
    """
    T = query.shape[0]
    H, D, qpk = p.num_heads, p.head_size, p.queries_per_kv
    out = torch.full((T, H * D), float("nan"), dtype=F64)
    q_all = query.to(F64).view(T, H, D)
    qlens = lengths_from_cu(cu_seqlens_q)
    klens = lengths_from_cu(cu_seqlens_k)
    window = _window(p, drop_window_with_alibi)
    wanted = None if rows is None else set(int(r) for r in rows)
    for b, (qb, Lb) in enumerate(zip(qlens, klens)):
        assert 0 <= qb <= Lb, "a subquery cannot be longer than its sequence"
        start = int(cu_seqlens_q[b])
        ts = [t for t in range(qb) if wanted is None or start + t in wanted]
        if not ts:
            continue
        cb = Lb - qb
        K, V = gather_kv(kv_cache, block_tables[b], Lb, p)
        pos = [cb + t for t in ts]
        idx = [start + t for t in ts]
        for h in range(H):
            g = kv_head_of(h, qpk)
            o = attend_rows(q_all[idx, h], pos, K[:, g], V[:, g], p.scale,
                            _slope(p, h), window, p.causal)
            out[idx, h * D:(h + 1) * D] = o
    return out


# ---------------------------------------------------------------------------
# a5, a6: block moves
# ---------------------------------------------------------------------------

def _check_pairs(pairs) -> list[tuple[int, int]]:
    pl = [(int(s), int(d)) for s, d in pairs]
    dsts = [d for _, d in pl]
    assert len(set(dsts)) == len(dsts), "destination blocks must be unique"
    return pl


def kv_copy_blocks(kv_caches: Sequence[torch.Tensor], pairs) -> None:
    """Copy block s to block d, K and V halves, in every layer's cache.

    xformers.py XFormersBackend.copy_blocks(kv_caches, src_to_dists): one
    source block may fan out to several destinations (copy-on-write forks).
    Reading taken: destinations are unique and are never also a source.
    """
    pl = _check_pairs(pairs)
    srcs = {s for s, _ in pl}
    assert not srcs & {d for _, d in pl}, "a destination is also a source"
    for cache in kv_caches:
        c = cache.view(torch.int16)
        for s, d in pl:
            c[:, d].copy_(c[:, s])


def kv_swap_blocks(src_cache: torch.Tensor, dst_cache: torch.Tensor,
                   pairs) -> None:
    """dst[:, d] = src[:, s] for every pair, across two caches.

    xformers.py XFormersBackend.swap_blocks(src_kv_cache, dst_kv_cache,
    src_to_dst): a one-way block move between two caches (device and host).
    """
    pl = _check_pairs(pairs)
    s16 = src_cache.view(torch.int16)
    d16 = dst_cache.view(torch.int16)
    for s, d in pl:
        d16[:, d].copy_(s16[:, s])
