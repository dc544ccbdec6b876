"""The pins catch plausible mistakes: each test plants one mistake in the
oracle (on the CPU, through monkeypatch) and checks that at least one pin
now fails."""
import numpy as np
import pytest

import test_oracle_attention as A
import test_oracle_formats as F
import test_oracle_pack as P
from oracle import attention, formats, pack


def fails(*checks):
    for c in checks:
        try:
            c()
        except AssertionError:
            return True
    return False


def test_swapped_nibble_order(monkeypatch):
    real = pack.pack_rows

    def mutated(latent, rope):
        row = real(latent, rope)
        b = row[:, :256]
        row[:, :256] = (b >> 4) | ((b & 15) << 4)
        return row

    monkeypatch.setattr(pack, "pack_rows", mutated)
    assert fails(P.check_hand_row)


def test_wrong_scale_divisor(monkeypatch):
    real = formats.e4m3_encode_quotient
    monkeypatch.setattr(formats, "e4m3_encode_quotient", lambda num, den: real(num, 4.0))
    assert fails(P.check_hand_row, F.check_scale_encode_all_bf16)


def test_unrounded_scale_in_quantiser(monkeypatch):
    """Quantising with amax/6 instead of the stored scale."""
    def mutated(latent, rope):
        latent = np.asarray(latent, dtype=np.float64)
        rope = np.asarray(rope, dtype=np.float64)
        row = np.zeros((latent.shape[0], 352), dtype=np.uint8)
        amax = np.abs(latent).reshape(-1, 32, 16).max(-1)
        S = np.repeat(amax / 6.0, 16, axis=1)
        codes = formats.e2m1_encode_scaled(latent, S)
        row[:, :256] = codes[:, 0::2] | (codes[:, 1::2] << 4)
        row[:, 256:288] = pack.group_scales(latent)
        row[:, 288:] = formats.e4m3_encode(rope)
        return row

    monkeypatch.setattr(pack, "pack_rows", mutated)
    assert fails(P.check_hand_row)


def test_dropped_sign_of_zero(monkeypatch):
    real = formats.e2m1_encode_scaled

    def mutated(x, scale):
        c = real(x, scale)
        return np.where((c & 7) == 0, np.uint8(0), c).astype(np.uint8)

    monkeypatch.setattr(formats, "e2m1_encode_scaled", mutated)
    assert fails(P.check_hand_row)


def test_ties_away_from_zero(monkeypatch):
    def mutated(x, scale):
        x = np.asarray(x, dtype=np.float64)
        scale = np.broadcast_to(np.asarray(scale, dtype=np.float64), x.shape)
        dist = np.abs(np.abs(x)[..., None] - scale[..., None] * formats.E2M1_TABLE[:8])
        # last minimum: ties go to the larger code
        mag = 7 - np.argmin(dist[..., ::-1], axis=-1)
        mag = np.where(scale == 0, 0, mag).astype(np.uint8)
        return (mag | np.where(np.signbit(x), 8, 0)).astype(np.uint8)

    monkeypatch.setattr(formats, "e2m1_encode_scaled", mutated)
    assert fails(F.check_e2m1_encode_exhaustive)
    assert fails(P.check_hand_row)


def test_wrong_e4m3_bias(monkeypatch):
    bad = np.array([formats.e4m3_value(c) * 0.5 for c in range(256)])
    monkeypatch.setattr(formats, "E4M3_TABLE", bad)
    assert fails(A.check_brute_force, P.check_hand_row)


def _attend_variant(kind):
    def f(q_lat, q_rope, K_lat, K_rope, sm_scale):
        H = q_lat.shape[0]
        if K_lat.shape[0] == 0:
            return np.zeros((H, K_lat.shape[1])), np.full(H, -np.inf)
        if kind == "no_rope":
            s = sm_scale * (q_lat @ K_lat.T)
        else:
            s = sm_scale * (q_lat @ K_lat.T + q_rope @ K_rope.T)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        L = e.sum(axis=1, keepdims=True)
        lse = (m + np.log(L))[:, 0]
        if kind == "log2":
            lse = (m + np.log2(L))[:, 0]
        out = (e / L) @ K_lat
        if kind == "unnormalised":
            out = e @ K_lat
        return out, lse
    return f


@pytest.mark.parametrize("kind,checks", [
    ("no_rope", ("check_brute_force",)),
    ("log2", ("check_equal_scores", "check_brute_force")),
    ("unnormalised", ("check_equal_scores", "check_brute_force")),
])
def test_attention_mistakes(monkeypatch, kind, checks):
    monkeypatch.setattr(attention, "attend", _attend_variant(kind))
    assert fails(*[getattr(A, c) for c in checks])


def test_negative_index_read_as_python_index(monkeypatch):
    real = attention.select_rows

    def mutated(topk_row, seq, block_table, seq_len, num_slots):
        p = np.asarray(topk_row, dtype=np.int64)
        p = np.where(p == -1, seq_len - 1, p)  # -1 taken as "last position"
        return real(p, seq, block_table, seq_len, num_slots)

    monkeypatch.setattr(attention, "select_rows", mutated)
    assert fails(A.check_padding)


def test_transposed_page_offset(monkeypatch):
    def mutated(topk_row, seq, block_table, seq_len, num_slots):
        p = np.asarray(topk_row, dtype=np.int64)
        limit = min(int(seq_len), block_table.shape[1] * 64)
        valid = (p >= 0) & (p < limit)
        pv = p[valid]
        slots = block_table[seq, pv % block_table.shape[1]].astype(np.int64) * 64 + pv // block_table.shape[1]
        return slots, int(((~valid) & (p != -1)).sum())

    monkeypatch.setattr(attention, "select_rows", mutated)
    assert fails(A.check_brute_force)


def test_missing_saturation(monkeypatch):
    """Nearest-grid search without the explicit saturation rule: float64
    distances far beyond 6*S all round to |x| and the search picks code 0."""
    def mutated(x, scale):
        x = np.asarray(x, dtype=np.float64)
        scale = np.broadcast_to(np.asarray(scale, dtype=np.float64), x.shape)
        dist = np.abs(np.abs(x)[..., None] - scale[..., None] * formats.E2M1_TABLE[:8])
        mag = formats._nearest_even(dist).astype(np.uint8)
        mag = np.where(scale == 0, 0, mag).astype(np.uint8)
        return (mag | np.where(np.signbit(x), 8, 0)).astype(np.uint8)

    monkeypatch.setattr(formats, "e2m1_encode_scaled", mutated)
    assert fails(F.check_e2m1_encode_exhaustive)


# ---- the top-k list builder, the multi-layer cache and the FP8 cache

import test_oracle_fp8cache as FC  # noqa: E402
import test_oracle_layered as LY  # noqa: E402
import test_oracle_topk as TK  # noqa: E402
from oracle import fp8cache, layered, topk  # noqa: E402


def _topk_variant(kind):
    def f(scores, k, lengths=None):
        s = np.asarray(scores, dtype=np.float64)
        T, ncols = s.shape
        out = np.full((T, k), -1, dtype=np.int64)
        for t in range(T):
            L = ncols if (lengths is None or kind == "lengths_ignored") else int(min(max(int(lengths[t]), 0), ncols))
            kk = min(k, L)
            pos = np.arange(L)
            if kind == "raw_bits":  # -0.0 ranked below +0.0, as its bit pattern does
                b = s[t, :L].astype(np.float32).view(np.uint32).astype(np.int64)
                key = np.where(b & 0x80000000, 0xFFFFFFFF - b, b | 0x80000000)
                order = np.lexsort((pos, -key))
            elif kind == "ties_high":
                order = np.lexsort((-pos, -(s[t, :L] + 0.0)))
            else:
                order = np.lexsort((pos, -(s[t, :L] + 0.0)))
            chosen = pos[order[:kk]]
            out[t, :kk] = chosen if kind == "unsorted" else np.sort(chosen)
        return out
    return f


@pytest.mark.parametrize("kind,checks", [
    ("ties_high", (TK.test_equal_scores_take_the_lowest_positions, lambda: TK.test_agrees_with_heapq(1))),
    ("unsorted", (TK.test_increasing_scores_take_the_last_positions, TK.test_chosen_scores_dominate_the_rest)),
    ("raw_bits", (TK.test_negative_zero_ties_with_positive_zero,)),
    ("lengths_ignored", (TK.test_short_lists_are_padded,)),
])
def test_topk_mistakes(monkeypatch, kind, checks):
    monkeypatch.setattr(topk, "topk_select", _topk_variant(kind))
    assert fails(*checks)


def test_layer_off_by_one(monkeypatch):
    real = layered.layer_view
    monkeypatch.setattr(layered, "layer_view", lambda cache, layer: real(cache, (layer + 1) % cache.shape[1]))
    assert fails(LY.test_rows_sit_at_the_layout_formula, LY.test_layered_decode_is_the_one_layer_decode)


def test_token_major_row_formula(monkeypatch):
    monkeypatch.setattr(layered, "row_byte_offset",
                        lambda block, layer, token, num_layers: ((block * 64 + token) * num_layers + layer) * 352)
    assert fails(LY.test_rows_sit_at_the_layout_formula)


def test_pack_writes_every_layer(monkeypatch):
    def mutated(latent, rope, slot_mapping, cache, layer):
        one = layered.layer_view(cache, layer)
        pack.pack_into_cache(latent, rope, slot_mapping, one)
        cache[:] = one[:, None]
        return cache

    monkeypatch.setattr(layered, "pack_into_layered_cache", mutated)
    assert fails(LY.test_packing_a_layer_leaves_the_others_alone)


def test_fp8_row_halves_swapped(monkeypatch):
    def mutated(latent, rope):
        row = np.empty((np.asarray(latent).shape[0], 576), dtype=np.uint8)
        row[:, :64] = formats.e4m3_encode(np.asarray(rope, dtype=np.float64))
        row[:, 64:] = formats.e4m3_encode(np.asarray(latent, dtype=np.float64))
        return row

    monkeypatch.setattr(fp8cache, "pack_rows", mutated)
    assert fails(FC.test_exact_values_round_trip)


def test_fp8_nan_instead_of_saturation(monkeypatch):
    real = fp8cache.pack_rows

    def mutated(latent, rope):
        row = real(latent, rope)
        vals = np.concatenate([np.asarray(latent, dtype=np.float64), np.asarray(rope, dtype=np.float64)], axis=1)
        over = np.abs(vals) > 448
        return np.where(over, np.where(vals < 0, 0xFF, 0x7F), row).astype(np.uint8)

    monkeypatch.setattr(fp8cache, "pack_rows", mutated)
    assert fails(FC.test_saturation)


def test_topk_variant_without_a_mistake_passes_every_pin(monkeypatch):
    # (the control: the mutations above fail the pins for their mistake, not
    # for a difference in how the variant is written)
    monkeypatch.setattr(topk, "topk_select", _topk_variant("none"))
    checks = [TK.test_equal_scores_take_the_lowest_positions, TK.test_increasing_scores_take_the_last_positions,
              TK.test_short_lists_are_padded, TK.test_chosen_scores_dominate_the_rest,
              TK.test_negative_zero_ties_with_positive_zero] + [lambda s=s: TK.test_agrees_with_heapq(s) for s in (1, 2, 3)]
    assert not fails(*checks)
