"""GPU parity of the staged baseline: stage 1 (NVFP4 rows -> temporary FP8
rows) bit-exact with the oracle's requantisation, stage 2 (attention over
FP8 rows) within the attention tolerance of the oracle on the same FP8
rows. The staged result's distance to the exact oracle is only reported: the
requantisation to FP8 is lossy by construction."""
import numpy as np
import pytest
import torch

import parity
from nvfp4_sparse_mla_gb300 import workloads
from oracle import staged as ostaged

pytestmark = pytest.mark.gpu

IMPLS = ["auto", "mma"]


def _impl(lib, name):
    return {"auto": None, "mma": lib.IMPL_MMA, "tcgen05": lib.IMPL_TCGEN05}[name]


@pytest.mark.parametrize("name", ["tiny", "padded", "decode_point"])
@pytest.mark.parametrize("impl", IMPLS)
def test_staged(lib, cuda, name, impl):
    w = workloads.make(name)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    d = parity.device_inputs(w, cuda)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    buf, idx = lib.nvfp4_stage_dequant_fp8(cache, d["block_table"], d["topk_idx"], d["q_seq_idx"], d["seq_lens"],
                                           err_word=err)
    rbuf, ridx = ostaged.stage_dequant_fp8_fast(ref_cache, w.block_table, w.topk_idx, w.q_seq_idx, w.seq_lens)
    gidx = idx.cpu().numpy()
    assert np.array_equal(gidx, ridx)
    valid = ridx >= 0
    assert np.array_equal(buf.cpu().numpy()[valid], rbuf[valid])
    assert err.cpu().tolist() == [0, 0]
    out, lse = lib.sparse_mla_decode_fp8rows(d["q_latent"], d["q_rope"], buf, idx, w.sm_scale,
                                             impl=_impl(lib, impl))
    ro, rl = ostaged.decode_fp8rows(w.q_latent, w.q_rope, rbuf, ridx, w.sm_scale)
    parity.assert_close(out, lse, ro, rl, f"staged/{name}/{impl}")
    # report (not gated): distance of the staged path to the exact oracle
    eo, el, _ = parity.oracle_decode(w, ref_cache)
    o = out.float().cpu().double().numpy()
    print(f"staged {name}: max |out - exact| = {np.abs(o - eo).max():.3e}")


@pytest.mark.parametrize("name", ["padded", "decode_point"])
def test_staged_buffer_as_fp8_cache(lib, cuda, name):
    """Stage 2 on the tcgen05 kernel: the staging buffer read as a paged FP8
    cache (token t's rows are pages t * topk / 64 onwards, the list entries
    the row indices) gives the oracle's attention over the same FP8 rows."""
    w = workloads.make(name)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    d = parity.device_inputs(w, cuda)
    buf, idx = lib.nvfp4_stage_dequant_fp8(cache, d["block_table"], d["topk_idx"], d["q_seq_idx"], d["seq_lens"])
    rbuf, ridx = ostaged.stage_dequant_fp8_fast(ref_cache, w.block_table, w.topk_idx, w.q_seq_idx, w.seq_lens)
    ppt = w.topk // 64
    bt = torch.arange(w.T * ppt, dtype=torch.int32, device=cuda).view(w.T, ppt)
    qs = torch.arange(w.T, dtype=torch.int32, device=cuda)
    out, lse = lib.sparse_mla_decode_fp8cache(d["q_latent"], d["q_rope"], buf.view(w.T * ppt, 64, 576), bt, idx,
                                              w.sm_scale, q_seq_idx=qs)
    ro, rl = ostaged.decode_fp8rows(w.q_latent, w.q_rope, rbuf, ridx, w.sm_scale)
    parity.assert_close(out, lse, ro, rl, f"staged tcgen05/{name}")
