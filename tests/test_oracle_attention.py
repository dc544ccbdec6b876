"""Pins for the oracle's sparse attention (CPU only).

Closed forms (one selected row; all-equal scores; identical rows), the
padding rule (empty slots contribute nothing), a brute-force dense masked
attention computed by torch's scaled_dot_product_attention in float64 over
rows decoded through torch's float8 dtype and the printed E2M1 grid, and
invariants (order of the list; a duplicated slot weighs double).
"""
import math

import numpy as np
import pytest
import torch

import golden_io
from nvfp4_sparse_mla_gb300 import workloads
from oracle import attention, pack, staged

PAGE = 64


def small_problem(seed=0, T=3, H=4, ctx=256, k=40, num_seqs=2, pad=0.25):
    """Logical rows per sequence, a shuffled page table and a cache filled
    page by page from the logical rows (the inverse direction of a lookup)."""
    rng = np.random.default_rng(seed)
    pages_per = ctx // PAGE
    n_pages = num_seqs * pages_per + 3
    perm = rng.permutation(n_pages)[:num_seqs * pages_per].reshape(num_seqs, pages_per)
    lat = rng.standard_normal((num_seqs, ctx, 512)) * rng.lognormal(0, 0.5, 512)
    rope = rng.standard_normal((num_seqs, ctx, 64))
    lat = torch.tensor(lat).to(torch.bfloat16).double().numpy()
    rope = torch.tensor(rope).to(torch.bfloat16).double().numpy()
    logical = np.stack([pack.pack_rows(lat[b], rope[b]) for b in range(num_seqs)])  # [B, ctx, 352]
    cache = np.zeros((n_pages, PAGE, 352), dtype=np.uint8)
    for b in range(num_seqs):
        for j in range(pages_per):
            cache[perm[b, j]] = logical[b, j * PAGE:(j + 1) * PAGE]
    q_seq = rng.integers(0, num_seqs, T)
    seq_lens = np.array([ctx - 7 * b for b in range(num_seqs)])
    topk = np.stack([rng.permutation(seq_lens[q_seq[t]])[:k] for t in range(T)])
    topk = np.where(rng.random(topk.shape) < pad, -1, topk)
    ql = torch.tensor(rng.standard_normal((T, H, 512))).to(torch.bfloat16).double().numpy()
    qr = torch.tensor(rng.standard_normal((T, H, 64))).to(torch.bfloat16).double().numpy()
    return dict(q_latent=ql, q_rope=qr, cache=cache, block_table=perm.astype(np.int32),
                topk_idx=topk.astype(np.int32), q_seq_idx=q_seq.astype(np.int32),
                seq_lens=seq_lens.astype(np.int32), logical=logical, sm_scale=1 / math.sqrt(192))


def run(p, **over):
    kw = {k: p[k] for k in ("q_latent", "q_rope", "cache", "block_table", "topk_idx",
                            "sm_scale", "q_seq_idx", "seq_lens")}
    kw.update(over)
    return attention.sparse_mla_decode(**kw)


def dense_decode(rows):
    """Decode rows [..., 352] with torch's float8 view for the FP8 bytes and
    the printed E2M1 grid for the 4-bit codes."""
    grid = np.array(golden_io.layout()["e2m1_grid"])
    signed = np.concatenate([grid, -grid])
    r = torch.from_numpy(np.ascontiguousarray(rows))
    scale = r[..., 256:288].contiguous().view(torch.float8_e4m3fn).double().numpy()
    rope = r[..., 288:352].contiguous().view(torch.float8_e4m3fn).double().numpy()
    lo = signed[rows[..., :256] & 15]
    hi = signed[rows[..., :256] >> 4]
    codes = np.stack([lo, hi], axis=-1).reshape(*rows.shape[:-1], 512)
    lat = codes * np.repeat(scale, 16, axis=-1)
    return lat, rope


def brute_force(p):
    """Dense attention over every logical position of the token's sequence,
    with a boolean mask that admits the selected positions (one column per
    slot, so duplicates count per slot)."""
    T, H, _ = p["q_latent"].shape
    out = np.zeros((T, H, 512))
    lse = np.zeros((T, H))
    for t in range(T):
        b = p["q_seq_idx"][t]
        lat, rope = dense_decode(p["logical"][b])  # [ctx, 512], [ctx, 64]
        L = p["seq_lens"][b]
        sel = p["topk_idx"][t]
        keep = (sel >= 0) & (sel < L)
        cols = sel[keep]
        K = np.concatenate([lat[cols], rope[cols]], axis=1)
        V = lat[cols]
        q = np.concatenate([p["q_latent"][t], p["q_rope"][t]], axis=1)
        if len(cols) == 0:
            out[t], lse[t] = 0.0, -np.inf
            continue
        qt = torch.from_numpy(q)[None]
        Kt = torch.from_numpy(K)[None]
        Vt = torch.from_numpy(V)[None]
        o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=p["sm_scale"])[0]
        s = torch.from_numpy(q) @ torch.from_numpy(K).T * p["sm_scale"]
        out[t] = o.numpy()
        lse[t] = torch.logsumexp(s, dim=1).numpy()
    return out, lse


def check_brute_force(seed=0):
    p = small_problem(seed)
    o, l, _ = run(p)
    bo, bl = brute_force(p)
    assert np.allclose(o, bo, rtol=1e-10, atol=1e-12)
    assert np.allclose(l, bl, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force(seed):
    check_brute_force(seed)


def check_one_index():
    p = small_problem(3, T=2, k=1, pad=0.0)
    o, l, _ = run(p)
    for t in range(2):
        b, pos = p["q_seq_idx"][t], p["topk_idx"][t, 0]
        lat, rope = dense_decode(p["logical"][b][pos][None])
        assert np.array_equal(o[t], np.broadcast_to(lat[0], o[t].shape))
        s = p["sm_scale"] * (p["q_latent"][t] @ lat[0] + p["q_rope"][t] @ rope[0])
        assert np.allclose(l[t], s, rtol=0, atol=1e-12)


def test_one_index():
    check_one_index()


def check_equal_scores():
    p = small_problem(4, pad=0.3)
    p["q_latent"] = np.zeros_like(p["q_latent"])
    p["q_rope"] = np.zeros_like(p["q_rope"])
    o, l, _ = run(p)
    for t in range(p["topk_idx"].shape[0]):
        b = p["q_seq_idx"][t]
        sel = p["topk_idx"][t]
        sel = sel[sel >= 0]
        lat, _ = dense_decode(p["logical"][b][sel])
        assert np.allclose(o[t], lat.mean(0)[None], rtol=1e-12, atol=1e-12)
        assert np.allclose(l[t], math.log(len(sel)), rtol=0, atol=1e-12)


def test_equal_scores():
    check_equal_scores()


def test_identical_rows():
    p = small_problem(5, T=1, k=7, pad=0.0)
    b = p["q_seq_idx"][0]
    pos = p["topk_idx"][0, 0]
    p["topk_idx"][0, :] = pos  # seven copies of one position
    o, l, _ = run(p)
    lat, rope = dense_decode(p["logical"][b][pos][None])
    s = p["sm_scale"] * (p["q_latent"][0] @ lat[0] + p["q_rope"][0] @ rope[0])
    assert np.allclose(o[0], lat[0][None], rtol=1e-14, atol=1e-14)
    assert np.allclose(l[0], s + math.log(7), rtol=0, atol=1e-12)


def check_padding():
    p = small_problem(6, pad=0.0)
    o, l, bad = run(p)
    padded = np.concatenate([p["topk_idx"], -np.ones((p["topk_idx"].shape[0], 9), np.int32)], 1)
    rng = np.random.default_rng(0)
    perm = rng.permutation(padded.shape[1])
    o2, l2, bad2 = run(p, topk_idx=padded[:, perm])
    assert np.allclose(o2, o, rtol=1e-13, atol=1e-14) and np.allclose(l2, l, rtol=1e-13, atol=1e-13)
    assert bad == bad2 == 0
    o3, l3, _ = run(p, topk_idx=-np.ones_like(p["topk_idx"]))
    assert np.all(o3 == 0) and np.all(np.isneginf(l3))


def test_padding_contributes_nothing():
    check_padding()


def test_out_of_range_is_masked_and_counted():
    p = small_problem(7, T=2, pad=0.0)
    o, l, _ = run(p)
    t2 = p["topk_idx"].copy()
    L = p["seq_lens"][p["q_seq_idx"]]
    extra = np.stack([[L[t], L[t] + 1000, -2, -1] for t in range(2)]).astype(np.int32)
    o2, l2, bad = run(p, topk_idx=np.concatenate([t2, extra], 1))
    assert bad == 6
    assert np.allclose(o2, o, rtol=1e-13, atol=1e-14) and np.allclose(l2, l, rtol=1e-13, atol=1e-13)


def test_order_invariance():
    p = small_problem(8)
    o, l, _ = run(p)
    rng = np.random.default_rng(1)
    perm = rng.permutation(p["topk_idx"].shape[1])
    o2, l2, _ = run(p, topk_idx=p["topk_idx"][:, perm])
    assert np.allclose(o2, o, rtol=1e-12, atol=1e-13) and np.allclose(l2, l, rtol=1e-13, atol=1e-13)


def test_duplicate_weighs_double():
    """Listing a position twice equals adding ln 2 to its score: checked
    against an explicit softmax over the distinct rows."""
    p = small_problem(9, T=1, k=12, pad=0.0)
    b = p["q_seq_idx"][0]
    sel = p["topk_idx"][0]
    dup = np.concatenate([sel, sel[:1]])[None].astype(np.int32)
    o, l, _ = run(p, topk_idx=dup)
    lat, rope = dense_decode(p["logical"][b][sel])
    s = p["sm_scale"] * (p["q_latent"][0] @ lat.T + p["q_rope"][0] @ rope.T)
    s[:, 0] += math.log(2)
    w = np.exp(s - s.max(1, keepdims=True))
    ref = (w / w.sum(1, keepdims=True)) @ lat
    assert np.allclose(o[0], ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(l[0], np.log(np.exp(s).sum(1)), rtol=1e-12, atol=1e-12)


def test_tokens_subset_matches_full():
    p = small_problem(10, T=4)
    o, l, _ = run(p)
    o2, l2, _ = run(p, tokens=[3, 1])
    assert np.array_equal(o2, o[[3, 1]]) and np.array_equal(l2, l[[3, 1]])


def test_workload_inputs_run():
    """The shared input generator feeds the oracle (tiny workload)."""
    w = workloads.tiny()
    lat, rope, slots = w.all_written()
    cache = np.zeros((w.num_pages, PAGE, 352), dtype=np.uint8)
    pack.pack_into_cache(lat.double().numpy(), rope.double().numpy(), slots.numpy(), cache)
    o, l, bad = attention.sparse_mla_decode(w.q_latent, w.q_rope, cache, w.block_table,
                                            w.topk_idx, w.sm_scale, w.q_seq_idx, w.seq_lens)
    assert o.shape == (1, 16, 512) and bad == 0 and np.all(np.isfinite(l))


# ---------------------------------------------------------------- staged

def test_staged_exact_when_requantisation_is_exact():
    """With power-of-two scales and magnitudes <= 448 every E2M1 * S value is
    an E4M3 value, so the staged path equals the direct one."""
    p = small_problem(11)
    flat = p["cache"].reshape(-1, 352)
    rng = np.random.default_rng(2)
    flat[:, 256:288] = rng.choice([0x30, 0x38, 0x40, 0x48, 0x50], size=flat[:, 256:288].shape)
    p["logical"] = None
    o, l, _ = run(p)
    buf, idx = staged.stage_dequant_fp8(p["cache"], p["block_table"], p["topk_idx"],
                                        p["q_seq_idx"], p["seq_lens"])
    o2, l2 = staged.decode_fp8rows(p["q_latent"], p["q_rope"], buf, idx, p["sm_scale"])
    assert np.allclose(o2, o, rtol=1e-12, atol=1e-13) and np.allclose(l2, l, rtol=1e-12, atol=1e-12)


def test_staged_requantisation_matches_torch_float8():
    p = small_problem(12, T=2)
    buf, idx = staged.stage_dequant_fp8(p["cache"], p["block_table"], p["topk_idx"],
                                        p["q_seq_idx"], p["seq_lens"])
    buf2, idx2 = staged.stage_dequant_fp8_fast(p["cache"], p["block_table"], p["topk_idx"],
                                               p["q_seq_idx"], p["seq_lens"])
    assert np.array_equal(buf, buf2) and np.array_equal(idx, idx2)
    for t in range(2):
        b = p["q_seq_idx"][t]
        for k in range(idx.shape[1]):
            pos = p["topk_idx"][t, k]
            if pos < 0:
                assert idx[t, k] == -1
                continue
            lat, _ = dense_decode(p["logical"][b][pos][None])
            v = np.clip(lat[0], -448, 448).astype(np.float32)
            ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(buf[t, k, :512], ref)
            assert np.array_equal(buf[t, k, 512:], p["logical"][b][pos][288:352])


def test_sequence_index_outside_the_table_selects_nothing():
    """A token whose sequence index has no block-table row attends to
    nothing (out 0, lse -inf); each of its entries other than -1 counts as a
    bad index. Checked against a token of a valid sequence in the same call."""
    rng = np.random.default_rng(21)
    bt = np.arange(4, dtype=np.int64).reshape(1, 4)
    cache = rng.integers(0, 256, size=(4, 64, 352), dtype=np.uint8)
    cache[:, :, 256:288] = 0x30  # finite scales
    cache[:, :, 288:] = 0x38     # finite RoPE
    ql = rng.standard_normal((2, 16, 512))
    qr = rng.standard_normal((2, 16, 64))
    topk = np.array([[3, 17, -1, 200], [3, 17, -1, 200]], dtype=np.int64)
    out, lse, bad = attention.sparse_mla_decode(ql, qr, cache, bt, topk, 0.1, q_seq_idx=np.array([0, 2]),
                                           seq_lens=np.array([256]))
    assert bad == 3
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(lse[0]))
    ref_out, ref_lse, _ = attention.sparse_mla_decode(ql[:1], qr[:1], cache, bt, topk[:1], 0.1, seq_lens=np.array([256]))
    assert np.array_equal(out[0], ref_out[0]) and np.array_equal(lse[0], ref_lse[0])
