"""One layer of a block-major multi-layer cache on the GPU
("Prime Inference: Fast, Reliable Serving for Frontier Open Models", section
"Changing the layout to reduce fragmentation"): pack is bit-exact against the
oracle's layered writer, every other layer is left alone, and the decode of a
layer matches the oracle and equals, bit for bit, the one-layer decode of the
same rows (the kernels differ only in where a row's bytes are)."""
import numpy as np
import pytest
import torch

import parity
from nvfp4_sparse_mla_gb300 import workloads
from oracle import layered as olay

pytestmark = pytest.mark.gpu

NUM_LAYERS = 3


def layer_inputs(w, layer):
    """Layer `layer`'s rows: the workload's tokens, varied per layer by a
    fixed scale and a rotation of the RoPE part (inputs, not results)."""
    lat, rope, slots = w.all_written()
    lat = (lat.float() * (1.0 + 0.5 * layer)).to(torch.bfloat16)
    rope = torch.roll(rope, shifts=layer, dims=1)
    return lat, rope, slots


@pytest.fixture(scope="module")
def setup(lib, cuda):
    w = workloads.decode_point(seed=31, T=4, ctx=30_000)
    cache = torch.zeros((w.num_pages, NUM_LAYERS, 64, 352), dtype=torch.uint8, device=cuda)
    ref = np.zeros((w.num_pages, NUM_LAYERS, 64, 352), dtype=np.uint8)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    for l in range(NUM_LAYERS):
        lat, rope, slots = layer_inputs(w, l)
        lib.nvfp4_mla_pack_layered(lat.to(cuda), rope.to(cuda), slots.to(cuda), cache, l, err_word=err)
        olay.pack_into_layered_cache(lat.double().numpy(), rope.double().numpy(), slots.numpy().astype(np.int64),
                                     ref, l)
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    return w, cache, ref


def test_layered_pack_is_bit_exact(setup):
    _, cache, ref = setup
    got = cache.cpu().numpy()
    for l in range(NUM_LAYERS):
        assert np.array_equal(got[:, l], ref[:, l]), f"layer {l}"


def test_layered_pack_leaves_other_layers_alone(lib, cuda, setup):
    w, cache, _ = setup
    c = cache.clone()
    before = c.cpu().numpy()
    lat, rope, slots = layer_inputs(w, 5)
    lib.nvfp4_mla_pack_layered(lat.to(cuda), rope.to(cuda), slots.to(cuda), c, 1)
    after = c.cpu().numpy()
    assert np.array_equal(after[:, 0], before[:, 0]) and np.array_equal(after[:, 2], before[:, 2])
    assert not np.array_equal(after[:, 1], before[:, 1])


@pytest.mark.parametrize("impl", ["tcgen05", "mma"])
@pytest.mark.parametrize("layer", [0, 2])
def test_layered_decode(lib, cuda, setup, impl, layer):
    w, cache, ref = setup
    code = lib.IMPL_TCGEN05 if impl == "tcgen05" else lib.IMPL_MMA
    d = parity.device_inputs(w, cuda)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    out, lse = lib.sparse_mla_decode_layered(d["q_latent"], d["q_rope"], cache, layer, d["block_table"],
                                             d["topk_idx"], w.sm_scale, q_seq_idx=d["q_seq_idx"],
                                             seq_lens=d["seq_lens"], err_word=err, impl=code)
    ro, rl, _ = olay.sparse_mla_decode_layered(w.q_latent, w.q_rope, ref, layer, w.block_table, w.topk_idx,
                                               w.sm_scale, w.q_seq_idx, w.seq_lens)
    parity.assert_close(out, lse, ro, rl, f"layered {impl} layer {layer}")
    assert err.cpu().tolist() == [0, 0]
    # the same rows in a one-layer cache give the same bits
    one = cache[:, layer].contiguous()
    o1, l1 = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], one, d["block_table"], d["topk_idx"], w.sm_scale,
                                   q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"], impl=code)
    assert torch.equal(out, o1) and torch.equal(lse, l1)
