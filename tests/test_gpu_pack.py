"""GPU parity of nvfp4_mla_pack: cache bytes must equal the oracle's
bit for bit."""
import numpy as np
import pytest
import torch

import golden_io
from nvfp4_sparse_mla_gb300 import workloads
from oracle import pack as opack

pytestmark = pytest.mark.gpu


def run_pack(lib, dev, lat, rope, slots, num_pages, err=None):
    cache = torch.zeros((num_pages, 64, 352), dtype=torch.uint8, device=dev)
    lib.nvfp4_mla_pack(lat.to(dev), rope.to(dev), slots.to(dev), cache, err_word=err)
    return cache.cpu().numpy()


def oracle_rows(lat, rope):
    return opack.pack_rows(lat.double().numpy(), rope.double().numpy())


def test_hand_row(lib, cuda):
    h = golden_io.hand_row()
    lat = torch.tensor(h["latent"][None]).to(torch.bfloat16)
    rope = torch.tensor(h["rope"][None]).to(torch.bfloat16)
    cache = run_pack(lib, cuda, lat, rope, torch.tensor([5], dtype=torch.int32), 1)
    assert np.array_equal(cache[0, 5], h["row"])
    assert not cache[0, :5].any() and not cache[0, 6:].any()


def _all_finite_bf16():
    v = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    return v[torch.isfinite(v)]


def test_every_bf16_value_latent(lib, cuda):
    """Every finite bf16 value goes through the latent quantiser, in random
    groups and in groups of neighbouring magnitudes (values near saturation)."""
    v = _all_finite_bf16()
    g = torch.Generator().manual_seed(0)
    shuffled = v[torch.randperm(v.numel(), generator=g)]
    by_mag = v[torch.argsort(v.float().abs())]
    rows = []
    for src in (shuffled, by_mag):
        n = (src.numel() + 511) // 512 * 512
        pad = torch.zeros(n - src.numel(), dtype=torch.bfloat16)
        rows.append(torch.cat([src, pad]).view(-1, 512))
    lat = torch.cat(rows)
    rope = torch.zeros((lat.shape[0], 64), dtype=torch.bfloat16)
    slots = torch.arange(lat.shape[0], dtype=torch.int32)
    pages = (lat.shape[0] + 63) // 64
    cache = run_pack(lib, cuda, lat, rope, slots, pages).reshape(-1, 352)[:lat.shape[0]]
    ref = oracle_rows(lat, rope)
    diff = np.nonzero((cache != ref).any(axis=1))[0]
    assert diff.size == 0, f"{diff.size} rows differ, first {diff[:5]}"


def test_every_bf16_value_rope(lib, cuda):
    v = _all_finite_bf16()
    n = (v.numel() + 63) // 64 * 64
    rope = torch.cat([v, torch.zeros(n - v.numel(), dtype=torch.bfloat16)]).view(-1, 64)
    lat = torch.zeros((rope.shape[0], 512), dtype=torch.bfloat16)
    slots = torch.arange(rope.shape[0], dtype=torch.int32)
    cache = run_pack(lib, cuda, lat, rope, slots, (rope.shape[0] + 63) // 64).reshape(-1, 352)[:rope.shape[0]]
    ref = oracle_rows(lat, rope)
    assert np.array_equal(cache, ref)


def test_special_groups(lib, cuda):
    """All-zero, all-equal, single-outlier and exact-midpoint groups."""
    rng = np.random.default_rng(3)
    rows = []
    rows.append(np.zeros(512))
    rows.append(np.full(512, 1.5))
    rows.append(np.full(512, -0.0))
    x = rng.standard_normal(512)
    x[::16] *= 20.0
    rows.append(x)
    S = 2.0 ** rng.integers(-9, 8, 32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0])
    rows.append((mids[None, :] * S[:, None]).reshape(-1))
    lat = torch.tensor(np.stack(rows)).to(torch.bfloat16)
    rope = torch.tensor(rng.standard_normal((len(rows), 64)) * 100).to(torch.bfloat16)
    slots = torch.arange(len(rows), dtype=torch.int32)
    cache = run_pack(lib, cuda, lat, rope, slots, 1).reshape(-1, 352)[:len(rows)]
    assert np.array_equal(cache, oracle_rows(lat, rope))


def test_prefill_chunk_with_outliers(lib, cuda):
    """The write+read workload's pack call: 6144 tokens, 1% outliers x20,
    distinct random slots of a 140K-token cache."""
    lat, rope, slots = workloads.pack_chunk(seed=4, n=6144, num_pages=2188)
    cache = run_pack(lib, cuda, lat, rope, slots, 2188).reshape(-1, 352)
    ref = np.zeros_like(cache)
    ref[slots.numpy()] = oracle_rows(lat, rope)
    assert np.array_equal(cache, ref)


def test_strided_inputs(lib, cuda):
    """latent and rope as column slices of one [N, 576] tensor."""
    rng = np.random.default_rng(4)
    kv = torch.tensor(rng.standard_normal((300, 576))).to(torch.bfloat16)
    slots = torch.tensor(rng.permutation(5 * 64)[:300], dtype=torch.int32)
    kv_d = kv.to(cuda)
    cache = torch.zeros((5, 64, 352), dtype=torch.uint8, device=cuda)
    lib.nvfp4_mla_pack(kv_d[:, :512], kv_d[:, 512:], slots.to(cuda), cache)
    ref = np.zeros((5 * 64, 352), dtype=np.uint8)
    ref[slots.numpy()] = oracle_rows(kv[:, :512], kv[:, 512:])
    assert np.array_equal(cache.cpu().numpy().reshape(-1, 352), ref)


def test_skipped_and_bad_slots(lib, cuda):
    rng = np.random.default_rng(5)
    lat = torch.tensor(rng.standard_normal((6, 512))).to(torch.bfloat16)
    rope = torch.tensor(rng.standard_normal((6, 64))).to(torch.bfloat16)
    slots = torch.tensor([3, -1, 64, 128, -7, 127], dtype=torch.int32)  # 128 is beyond 2 pages
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    cache = run_pack(lib, cuda, lat, rope, slots, 2, err=err).reshape(-1, 352)
    ref = oracle_rows(lat, rope)
    assert np.array_equal(cache[3], ref[0]) and np.array_equal(cache[64], ref[2])
    assert np.array_equal(cache[127], ref[5])
    assert int((cache.any(axis=1)).sum()) == 3
    e = err.cpu().tolist()
    assert e[0] & 0x4 and e[1] == 1


def test_empty_is_noop(lib, cuda):
    cache = torch.zeros((1, 64, 352), dtype=torch.uint8, device=cuda)
    z = torch.zeros((0, 512), dtype=torch.bfloat16, device=cuda)
    lib.nvfp4_mla_pack(z, torch.zeros((0, 64), dtype=torch.bfloat16, device=cuda),
                       torch.zeros(0, dtype=torch.int32, device=cuda), cache)
    assert not cache.any()
