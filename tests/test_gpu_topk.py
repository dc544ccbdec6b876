"""The top-k list builder on the GPU against the oracle: exact lists (the
chosen set is unique once equal scores rank by position, and it is written in
increasing order), on the decode point's size, with heavy ties, with short
and empty candidate lists, and feeding the decode."""
import numpy as np
import pytest
import torch

import parity
from nvfp4_sparse_mla_gb300 import workloads
from oracle import topk as otopk

pytestmark = pytest.mark.gpu


def check(lib, cuda, s, k, lengths=None):
    d = torch.from_numpy(s.astype(np.float32)).to(cuda)
    dl = None if lengths is None else torch.tensor(lengths, dtype=torch.int32, device=cuda)
    got = lib.nvmla_topk_select(d, k, dl).cpu().numpy()
    want = otopk.topk_select(s.astype(np.float32), k, lengths)
    assert np.array_equal(got, want), f"first difference at {np.argwhere(got != want)[0].tolist()}"
    return got


def test_decode_point_size(lib, cuda):
    rng = np.random.default_rng(21)
    check(lib, cuda, rng.standard_normal((15, 200_000)), 2048)


def test_rows_longer_than_shared_memory_holds(lib, cuda):
    # 8 chunks of more than 32K keys: every pass reads the chunk from global
    # memory; one row also has its winners bunched
    rng = np.random.default_rng(29)
    s = rng.standard_normal((2, 320_003))
    s[1, 300_000:302_048] = 5.0
    check(lib, cuda, s, 2048)
    check(lib, cuda, s, 2048, lengths=[262_144, 262_148])


def test_longest_rows_kept_in_shared_memory(lib, cuda):
    # 262,144 scores: every CTA's eighth is exactly the 32,768 keys shared
    # memory holds (every copy round full, every walk's mask full); one more
    # column and the whole launch takes the global-memory kernel
    rng = np.random.default_rng(34)
    s = rng.standard_normal((2, 262_144))
    check(lib, cuda, s, 2048)
    check(lib, cuda, s, 2048, lengths=[262_144, 131_071])
    s1 = rng.standard_normal((2, 262_145))
    check(lib, cuda, s1, 2048)


def test_heavy_ties(lib, cuda):
    rng = np.random.default_rng(22)
    check(lib, cuda, rng.integers(0, 5, (6, 50_000)).astype(np.float64), 2048)
    check(lib, cuda, np.zeros((2, 10_000)), 2048)
    s = rng.standard_normal((3, 9000))
    s[:, ::3] = -0.0
    s[:, 1::3] = 0.0
    check(lib, cuda, s, 2048)


def test_ties_inside_the_pool(lib, cuda):
    # ~2,500 keys tied at the top value: the pool takes them all and the
    # list ends with the lowest 2,048 of their positions
    rng = np.random.default_rng(31)
    check(lib, cuda, rng.integers(0, 20, (3, 50_000)).astype(np.float64), 2048)
    # scores on a 0.001 grid: the threshold key has a few exact copies among
    # the last keys rank 0 counts
    check(lib, cuda, np.round(rng.standard_normal((3, 200_000)), 3), 2048)


def test_many_equal_keys_per_chunk(lib, cuda):
    # more keys in the chosen bin than rank 0's pool holds, and more per
    # thread than its list holds: the cluster-wide passes over the chunk
    check(lib, cuda, np.zeros((2, 200_000)), 2048)
    rng = np.random.default_rng(26)
    check(lib, cuda, rng.integers(0, 4, (3, 200_000)).astype(np.float64), 2048)


def test_winners_bunched_in_one_segment(lib, cuda):
    # the whole list in the last or first few warp segments of one CTA's
    # chunk (more kept keys than a warp holds: that CTA re-reads its chunk),
    # and 200 winners inside one segment (they fit)
    n = 200_000
    up = np.arange(n, dtype=np.float64)
    check(lib, cuda, np.stack([up, up[::-1].copy()]), 2048)
    rng = np.random.default_rng(27)
    s = rng.standard_normal((2, n))
    s[0, 51_000:51_200] = 10.0 + rng.random(200)
    s[1, 120_000:120_200] = 10.0
    check(lib, cuda, s, 2048)


def test_one_thread_with_many_candidates(lib, cuda):
    # spikes every 4096 positions land on one thread of every CTA, more of
    # them than the thread lists: the chunk is walked again for them
    rng = np.random.default_rng(30)
    s = rng.standard_normal((2, 200_000))
    for r in range(2):
        idx = np.arange(200_000)
        s[r, (idx + 1000 * r) % 4096 < 4] = 100.0 + rng.random(int(((idx + 1000 * r) % 4096 < 4).sum()))
    check(lib, cuda, s, 2048)


def test_one_chunk_lifts_the_cut(lib, cuda):
    # every 25th position of the first eighth of the row far above the rest:
    # that CTA's cut lies above them, fewer than k keys of the row do, and
    # the select falls back to the cluster-wide passes; a second row puts
    # 3,000 of them in one eighth (more than its list holds)
    rng = np.random.default_rng(32)
    s = rng.standard_normal((2, 200_000))
    s[0, 0:25_000:25] = 100.0 + rng.random(1000)
    s[1, 100_000:175_000:25] = 50.0 + rng.random(3000)
    check(lib, cuda, s, 2048)
    check(lib, cuda, s, 700)


def test_infinite_scores(lib, cuda):
    # +inf scores at scattered positions (fewer than k in one row, more
    # than k in another: ties at +inf taken by lowest position), a row that
    # is -inf but for 1,000 finite scores (so -inf ties fill the list), and
    # a row of +inf and -inf only
    rng = np.random.default_rng(33)
    s = rng.standard_normal((4, 200_000))
    s[0, rng.choice(200_000, 300, replace=False)] = np.inf
    s[1, rng.choice(200_000, 5_000, replace=False)] = np.inf
    s[2, :] = -np.inf
    s[2, rng.choice(200_000, 1_000, replace=False)] = rng.standard_normal(1_000)
    s[3, :] = np.where(rng.random(200_000) < 0.01, np.inf, -np.inf)
    check(lib, cuda, s, 2048)


def test_rows_not_16_byte_aligned(lib, cuda):
    rng = np.random.default_rng(28)
    s = rng.standard_normal((4, 40_001))
    check(lib, cuda, s, 2048)
    check(lib, cuda, s, 2048, lengths=[40_001, 40_000, 39_999, 2050])


def test_short_and_empty_lists(lib, cuda):
    rng = np.random.default_rng(23)
    s = rng.standard_normal((5, 4000))
    check(lib, cuda, s, 2048, lengths=[4000, 2048, 2047, 5, 0])
    check(lib, cuda, s, 2048, lengths=[9999, 3000, 1, 2049, 4000])
    check(lib, cuda, s[:, :1000], 2048)
    check(lib, cuda, s, 1)
    check(lib, cuda, s, 777)


def test_lists_feed_the_decode(lib, cuda):
    w = workloads.decode_point(seed=24, T=3, ctx=40_000)
    rng = np.random.default_rng(25)
    scores = rng.standard_normal((w.T, 40_000))
    lengths = [40_000, 30_000, 1_500]
    d = parity.device_inputs(w, cuda)
    tk = lib.nvmla_topk_select(torch.from_numpy(scores.astype(np.float32)).to(cuda), 2048,
                               torch.tensor(lengths, dtype=torch.int32, device=cuda))
    want = otopk.topk_select(scores.astype(np.float32), 2048, lengths)
    assert np.array_equal(tk.cpu().numpy(), want)
    cache = parity.device_cache(lib, w, cuda)
    out, lse = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], tk, w.sm_scale,
                                     q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"])
    ref_cache = parity.oracle_cache(w)
    ro, rl, _ = parity.oracle_decode(w, ref_cache, topk_idx=torch.from_numpy(want.astype(np.int32)))
    parity.assert_close(out, lse, ro, rl, "decode over selected lists")
