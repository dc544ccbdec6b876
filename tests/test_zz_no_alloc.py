"""sparse_mla_decode_noalloc: the decode call that allocates nothing and
keeps its split partials in the library's own device scratch.

It must give the same bits as sparse_mla_decode handed a workspace of the
default size (same kernels, same split count), on two calls in a row: the
second call finds the first call's partials in the scratch and must not
depend on them. The tcgen05 kernel (head counts that are multiples of 64)
combines its splits in shared memory and needs no scratch; the mma.sync
kernel (the other head counts) keeps fp32 partials there. The file name sorts
last so that it also runs after every other GPU test in the process."""
import ctypes

import pytest
import torch

import parity
from nvfp4_sparse_mla_gb300 import workloads

SCRATCH_BYTES = 16 << 20
SMS = 152  # the no-device model and a GB300


def _bound(T, H, sms=SMS):
    """The header's bound on the scratch a call needs: the mma.sync kernel
    keeps T * S * H * (512 + 2) fp32 values, and its split count S gives
    T * S <= floor(sms / ceil(H / 64)); head counts that are multiples of 64
    need none."""
    if H % 64 == 0:
        return 0
    return (sms // ((H + 63) // 64)) * H * 514 * 4


def test_scratch_size(lib):
    assert lib.sparse_mla_decode_noalloc_max_scratch() == SCRATCH_BYTES


@pytest.mark.skipif(torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != SMS,
                    reason="the bound is stated for 152 SMs")
def test_every_shape_within_the_stated_bound(lib):
    """Host-only sweep of every token count at every head count (top-2048):
    the scratch a call needs never exceeds the header's bound, which fits
    the 16 MiB scratch for every head count but 112."""
    for H in range(16, 129, 16):
        b = _bound(64, H)
        assert (b <= SCRATCH_BYTES) == (H != 112), H
        worst = 0
        for T in range(1, 65536):
            need = lib.sparse_mla_decode_workspace_size(T, H, 2048)
            assert need <= b, (T, H, need, b)
            worst = max(worst, need)
        assert worst == 0 if H % 64 == 0 else worst > 0, H


def test_rejects_shapes_beyond_the_scratch(lib):
    """Host-side: a shape whose default split scratch exceeds 16 MiB returns
    NVMLA_ERR_WORKSPACE with a message, before touching any pointer."""
    T, H, topk = 38, 112, 2048
    need = lib.sparse_mla_decode_workspace_size(T, H, topk)
    assert need > SCRATCH_BYTES
    L = lib.load()
    ok = ctypes.c_void_p(0x10000)  # never dereferenced: the size check fails first
    st = L.sparse_mla_decode_noalloc(ok, ok, ok, 10, ok, 1, 4, ok, topk, None, None, T, H, 0.1, ok, ok, None, None)
    assert st == 4
    msg = L.nvmla_last_error().decode()
    assert "sparse_mla_decode_noalloc" in msg and str(need) in msg and str(SCRATCH_BYTES) in msg


def test_binding_requires_outputs(lib):
    q = torch.zeros((1, 64, 512), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        lib.sparse_mla_decode_noalloc(q, torch.zeros((1, 64, 64), dtype=torch.bfloat16),
                                      torch.zeros((1, 64, 352), dtype=torch.uint8),
                                      torch.zeros((1, 1), dtype=torch.int32), torch.zeros((1, 1), dtype=torch.int32),
                                      0.1, None, torch.zeros((1, 64)))


def _inputs(w, dev):
    """Two different problems on the same cache: the workload's own queries,
    and the same queries with heads and top-k order reversed."""
    a = parity.device_inputs(w, dev)
    b = dict(a)
    b["q_latent"] = a["q_latent"].flip(1).contiguous()
    b["q_rope"] = a["q_rope"].flip(1).contiguous()
    b["topk_idx"] = a["topk_idx"].flip(1).contiguous()
    return a, b


def _reference(lib, w, cache, d):
    return lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"], w.sm_scale,
                                 q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"])


def _noalloc(lib, w, cache, d, out, lse, err):
    return lib.sparse_mla_decode_noalloc(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"],
                                         w.sm_scale, out, lse, q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"],
                                         err_word=err)


def _workload(name):
    if name == "h48_near_limit":
        # 15 tokens x 48 heads: the mma.sync kernel with 10 splits, 14.8 MB
        # of the 16 MiB scratch
        return workloads.decode_point(seed=21, T=15, H=48, ctx=20_000)
    return workloads.make(name)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["decode_point", "tiny", "h48_near_limit"])
def test_two_calls_match_sparse_mla_decode(lib, cuda, name):
    """decode_point runs the tcgen05 kernel with 8 splits combined in shared
    memory (no scratch); tiny (16 heads) and h48_near_limit (48 heads) run the
    mma.sync kernel with fp32 partials in the scratch and its merge kernel."""
    w = _workload(name)
    need = lib.sparse_mla_decode_workspace_size(w.T, w.H, w.topk_idx.shape[1])
    assert (need > 0) == (w.H % 64 != 0)
    assert need <= SCRATCH_BYTES
    if name == "h48_near_limit":
        assert need > (14 << 20)
    cache = parity.device_cache(lib, w, cuda)
    a, b = _inputs(w, cuda)
    ref_a = _reference(lib, w, cache, a)
    ref_b = _reference(lib, w, cache, b)
    outs = [torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=cuda) for _ in range(3)]
    lses = [torch.empty((w.T, w.H), dtype=torch.float32, device=cuda) for _ in range(3)]
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    # warm-up: loads the library's code and looks up the scratch
    _noalloc(lib, w, cache, a, outs[2], lses[2], err)
    torch.cuda.synchronize()
    # nothing else allocates between the two readings: this process's torch
    # allocator (memory_allocated) and the device (free bytes) must not move
    allocated = torch.cuda.memory_allocated(cuda)
    free_before = torch.cuda.mem_get_info(cuda)[0]
    launches = lib.launch_count()
    _noalloc(lib, w, cache, a, outs[0], lses[0], err)
    _noalloc(lib, w, cache, b, outs[1], lses[1], err)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated(cuda) == allocated, "the calls allocated through torch"
    assert torch.cuda.mem_get_info(cuda)[0] == free_before, "the calls changed the device's free memory"
    assert lib.launch_count() - launches == (2 if w.H % 64 == 0 else 4)  # per call: decode (+ merge)
    assert err.tolist() == [0, 0]
    assert torch.equal(outs[0], ref_a[0]) and torch.equal(lses[0], ref_a[1]), "first call differs"
    assert torch.equal(outs[1], ref_b[0]) and torch.equal(lses[1], ref_b[1]), "second call differs"
    assert not torch.equal(outs[0], outs[1]), "the two problems should give different outputs"
