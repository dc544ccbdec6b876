"""The FP8 cache (576-byte E4M3 rows) on the GPU: its pack is bit-exact
against the oracle, and the tcgen05 decode over it matches the oracle's FP8
decode within the decode tolerance, for several split counts."""
import numpy as np
import pytest
import torch

import parity
from nvfp4_sparse_mla_gb300 import workloads
from oracle import fp8cache as ofp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup(lib, cuda):
    w = workloads.decode_point(seed=41, T=3, ctx=20_000)
    lat, rope, slots = w.all_written()
    cache = torch.zeros((w.num_pages, 64, 576), dtype=torch.uint8, device=cuda)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    lib.fp8_mla_pack(lat.to(cuda), rope.to(cuda), slots.to(cuda), cache, err_word=err)
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    return w, cache


def test_fp8_pack_is_bit_exact(setup):
    w, cache = setup
    lat, rope, slots = w.all_written()
    pick = np.random.default_rng(0).choice(slots.shape[0], 1500, replace=False)
    want = ofp8.pack_rows(lat[pick].double().numpy(), rope[pick].double().numpy())
    got = cache.reshape(-1, 576).cpu().numpy()[slots.numpy()[pick]]
    assert np.array_equal(got, want)


def oracle_cache_for(w):
    """The oracle's FP8 cache holding the rows the tokens select."""
    lat, rope, slots = w.all_written()
    bt, L = w.block_table.numpy(), w.seq_lens.numpy()
    need = set()
    for t in range(w.T):
        b = int(w.q_seq_idx[t])
        p = w.topk_idx[t].numpy().astype(np.int64)
        p = p[(p >= 0) & (p < L[b])]
        need.update((bt[b, p // 64].astype(np.int64) * 64 + p % 64).tolist())
    s = slots.numpy().astype(np.int64)
    keep = np.isin(s, np.fromiter(need, dtype=np.int64))
    c = np.zeros((w.num_pages, 64, 576), dtype=np.uint8)
    ofp8.pack_into_cache(lat[keep].double().numpy(), rope[keep].double().numpy(), s[keep], c)
    return c


@pytest.mark.parametrize("splits", [None, 1, 3, 8])
def test_fp8_cache_decode(lib, cuda, setup, splits):
    w, cache = setup
    ref = oracle_cache_for(w)
    ro, rl, _ = ofp8.sparse_mla_decode(w.q_latent, w.q_rope, ref, w.block_table, w.topk_idx, w.sm_scale,
                                       w.q_seq_idx, w.seq_lens)
    d = parity.device_inputs(w, cuda)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    out, lse = lib.sparse_mla_decode_fp8cache(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"],
                                              w.sm_scale, q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"],
                                              err_word=err, num_splits=splits)
    parity.assert_close(out, lse, ro, rl, f"fp8 cache splits={splits}")
    assert err.cpu().tolist() == [0, 0]


def test_fp8_cache_needs_64_heads(lib, cuda, setup):
    w, cache = setup
    q = torch.zeros((1, 16, 512), dtype=torch.bfloat16, device=cuda)
    qr = torch.zeros((1, 16, 64), dtype=torch.bfloat16, device=cuda)
    with pytest.raises(lib.NvmlaError) as e:
        lib.sparse_mla_decode_fp8cache(q, qr, cache, w.block_table.to(cuda), w.topk_idx[:1].to(cuda), 0.1)
    assert e.value.status == 2
