"""The NVMLA_DEBUG_BOUNDS build of the library: the same sources compiled with
every data-dependent index of the tcgen05 decode kernel (cache rows,
block-table and slot-list entries, output positions, tile and split counts)
checked against its buffer, a failure recorded as NVMLA_ERRW_BOUNDS in
err_word. On the workloads' shapes, at the extreme split counts, with two
head blocks, with padded lists and over the FP8 cache it records nothing,
and its outputs still match the oracle. (Its shared-memory and TMEM offsets
are checked exhaustively on the host: test_layout_bounds.py.)"""
import numpy as np
import pytest
import torch

import parity
from nvfp4_sparse_mla_gb300 import _build, workloads
from oracle import fp8cache as ofp8

pytestmark = pytest.mark.gpu

ERRW_BOUNDS = 0x10


@pytest.fixture(scope="module")
def debug_lib(lib, cuda, tmp_path_factory):
    """The binding, pointed at a NVMLA_DEBUG_BOUNDS build for this module."""
    d = tmp_path_factory.mktemp("debug_bounds")
    path = _build.build(out_dir=str(d), lib=str(d / "libnvmla_debug_bounds.so"), defines=("NVMLA_DEBUG_BOUNDS",))
    saved_lib, saved_path = lib._lib, lib.library_path
    lib._lib = None
    lib.library_path = lambda: path
    lib.load()
    assert lib.build_flags() & lib.BUILD_DEBUG_BOUNDS, "the variant was not built with the checks"
    yield lib
    lib._lib, lib.library_path = saved_lib, saved_path


def _workload(name):
    if name == "two_head_blocks":
        return workloads.decode_point(seed=51, T=3, H=128, ctx=20_000)
    if name == "short_list":
        return workloads.decode_point(seed=52, T=4, ctx=9_000, topk=300)
    return workloads.make(name)


@pytest.mark.parametrize("name,splits", [("decode_point", None), ("decode_point", 1), ("decode_point", 16),
                                         ("padded", None), ("two_head_blocks", 3), ("short_list", None)])
def test_nvfp4_decode_records_no_bound_failure(debug_lib, cuda, name, splits):
    w = _workload(name)
    cache = parity.device_cache(debug_lib, w, cuda)
    d = parity.device_inputs(w, cuda)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    out, lse = debug_lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"],
                                           w.sm_scale, q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"],
                                           err_word=err, impl=debug_lib.IMPL_TCGEN05, num_splits=splits)
    torch.cuda.synchronize()
    e = err.cpu().tolist()
    assert e[0] & ERRW_BOUNDS == 0, e
    assert e == [0, 0], e
    toks = list(range(min(w.T, 6)))
    ref = parity.oracle_cache(w, tokens=toks)
    ro, rl, _ = parity.oracle_decode(w, ref, tokens=toks)
    parity.assert_close(out[toks], lse[toks], ro, rl, f"debug bounds {name} splits={splits}")


def test_fp8_decode_records_no_bound_failure(debug_lib, cuda):
    w = workloads.decode_point(seed=53, T=3, ctx=20_000)
    lat, rope, slots = w.all_written()
    cache = torch.zeros((w.num_pages, 64, 576), dtype=torch.uint8, device=cuda)
    debug_lib.fp8_mla_pack(lat.to(cuda), rope.to(cuda), slots.to(cuda), cache)
    d = parity.device_inputs(w, cuda)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    out, lse = debug_lib.sparse_mla_decode_fp8cache(d["q_latent"], d["q_rope"], cache, d["block_table"],
                                                    d["topk_idx"], w.sm_scale, q_seq_idx=d["q_seq_idx"],
                                                    seq_lens=d["seq_lens"], err_word=err)
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    c = np.zeros((w.num_pages, 64, 576), dtype=np.uint8)
    ofp8.pack_into_cache(lat.double().numpy(), rope.double().numpy(), slots.numpy().astype(np.int64), c)
    ro, rl, _ = ofp8.sparse_mla_decode(w.q_latent, w.q_rope, c, w.block_table, w.topk_idx, w.sm_scale,
                                       w.q_seq_idx, w.seq_lens)
    parity.assert_close(out, lse, ro, rl, "debug bounds fp8 cache")


def test_bad_entries_are_still_masked_not_bound_failures(debug_lib, cuda):
    """Out-of-range list entries are the data's problem (NVMLA_ERRW_BAD_INDEX),
    masked before any index is formed: the bounds checks see none of them."""
    w = workloads.decode_point(seed=54, T=2, ctx=9_000, topk=256)
    cache = parity.device_cache(debug_lib, w, cuda)
    d = parity.device_inputs(w, cuda)
    tk = d["topk_idx"].clone()
    tk[0, :7] = torch.tensor([9_000, 10**9, -2, -5, 2**31 - 1, 9_001, -(2**31)], dtype=torch.int32)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    debug_lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], tk, w.sm_scale,
                                q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"], err_word=err,
                                impl=debug_lib.IMPL_TCGEN05)
    torch.cuda.synchronize()
    e = err.cpu().tolist()
    assert e[0] & ERRW_BOUNDS == 0, e
    assert e[0] & 0x1 and e[1] == 7, e
