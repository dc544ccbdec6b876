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


def test_heavy_ties(lib, cuda):
    rng = np.random.default_rng(22)
    check(lib, cuda, rng.integers(0, 5, (6, 50_000)).astype(np.float64), 2048)
    check(lib, cuda, np.zeros((2, 10_000)), 2048)
    s = rng.standard_normal((3, 9000))
    s[:, ::3] = -0.0
    s[:, 1::3] = 0.0
    check(lib, cuda, s, 2048)


def test_many_equal_keys_per_chunk(lib, cuda):
    # more equal keys in the chosen bin than a CTA keeps in shared memory
    check(lib, cuda, np.zeros((2, 200_000)), 2048)
    rng = np.random.default_rng(26)
    check(lib, cuda, rng.integers(0, 4, (3, 200_000)).astype(np.float64), 2048)


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
