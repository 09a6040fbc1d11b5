"""Planted mistakes in the oracle must each break at least one pin.

Every mutation below is a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand); it is applied to the CPU oracle
with monkeypatch, never to the CUDA path.
"""
import math

import pytest
import torch

import oracle.paged_attention as OP
from oracle_pins import ALL_PINS

_orig_attend = OP.attend_rows


def _attend_variant(drop_scale=False, drop_causal=False, swap_kv=False):
    def attend(q, positions, K, V, scale, slope, window, causal=True):
        if swap_kv:
            K, V = V, K
        if drop_scale:
            scale = 1.0
        if not drop_causal:
            return _orig_attend(q, positions, K, V, scale, slope, window, causal)
        n = q.shape[0]
        out = torch.zeros(n, V.shape[1], dtype=torch.float64)
        for r in range(n):
            i = int(positions[r])
            s = scale * (K @ q[r])
            if slope is not None:
                s = s + OP.alibi_bias(slope, torch.arange(K.shape[0]), i)
            out[r] = torch.softmax(s, 0) @ V
        return out
    return attend


MUTATIONS = {
    "gqa_modulo": ("kv_head_of", lambda h, qpk: h % 2),
    "gqa_identity": ("kv_head_of", lambda h, qpk: 0),
    "alibi_sign": ("alibi_bias", lambda a, j, i: a * (i - j)),
    "alibi_dropped": ("alibi_bias", lambda a, j, i: 0.0 * (j - i)),
    "alibi_double": ("alibi_bias", lambda a, j, i: 2 * a * (j - i)),
    "window_one_too_wide": ("window_lo",
                            lambda i, w: max(0, i - w) if w > 0 else 0),
    "window_one_too_narrow": ("window_lo",
                              lambda i, w: max(0, i - w + 2) if w > 0 else 0),
    "decode_position_off": ("decode_position", lambda L: max(0, L - 2)),
    "slot_swapped": ("slot_location", lambda s, bs: (s % bs, s // bs)),
    "slot_off_by_one": ("slot_location", lambda s, bs: ((s + 1) // bs, (s + 1) % bs)),
    "scale_dropped": ("attend_rows", _attend_variant(drop_scale=True)),
    "causal_dropped": ("attend_rows", _attend_variant(drop_causal=True)),
    "k_v_swapped": ("attend_rows", _attend_variant(swap_kv=True)),
    "cu_shifted": ("lengths_from_cu",
                   lambda cu: [int(cu[k + 1]) - int(cu[0])
                               for k in range(len(cu) - 1)]),
    "combine_unweighted": ("combine_split_partials",
                           lambda parts: sum(o for o, _, _ in parts) / len(parts)),
}


def _gather_wrong_block(kv_cache, table_row, n_tokens, p):
    # logical block k read from table entry (k + 1) mod nblocks
    nb = (n_tokens + p.block_size - 1) // p.block_size
    rot = torch.tensor([int(table_row[(k + 1) % nb]) for k in range(nb)])
    return _orig_gather(kv_cache, rot, n_tokens, p)


_orig_gather = OP.gather_kv
MUTATIONS["block_table_rotated"] = ("gather_kv", _gather_wrong_block)


def _attend_always_causal(q, positions, K, V, scale, slope, window, causal=True):
    # the non-causal flag ignored: encoder attention would lose its future keys
    return _orig_attend(q, positions, K, V, scale, slope, window, True)


MUTATIONS["noncausal_ignored"] = ("attend_rows", _attend_always_causal)
# speculative tokens placed one position too early / counted from the front
MUTATIONS["multi_position_off"] = ("multi_decode_position", lambda L, q, t: L - q + t - 1)
MUTATIONS["multi_position_front"] = ("multi_decode_position", lambda L, q, t: t)
# decode context parallelism: ranks' tokens placed contiguously, or miscounted
MUTATIONS["dcp_position_block"] = ("dcp_global_position", lambda k, R, r: r * 5 + k)
MUTATIONS["dcp_local_len_floor"] = ("dcp_local_seq_len", lambda L, R, r: (L - r) // R if L > r else 0)


def _encode_truncating(x):
    # rounds toward zero instead of to nearest
    if x != x:
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = min(abs(x), 448.0)
    best = 0
    for c, v in enumerate(OP._E4M3_POS):
        if v <= a:
            best = c
    return sign | best


MUTATIONS["fp8_truncating"] = ("e4m3_encode", _encode_truncating)
MUTATIONS["fp8_scale_ignored"] = ("_dequant", lambda codes, scale: OP._E4M3_TABLE[codes.to(torch.int64)])


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_mutation_is_caught(mutation, monkeypatch):
    attr, fn = MUTATIONS[mutation]
    monkeypatch.setattr(OP, attr, fn)
    failed = []
    for name, pin in ALL_PINS.items():
        try:
            pin()
        except Exception:
            failed.append(name)
    assert failed, f"mutation {mutation} broke no pin"
