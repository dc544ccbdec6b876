"""Helpers shared by the GPU parity tests: put a synthetic workload on the
device through the library's own pack call, and build the oracle's reference
from the same seeded inputs (never from anything the CUDA path produced)."""
import numpy as np
import torch

from nvfp4_sparse_mla_gb300 import workloads
from oracle import attention as oatt
from oracle import pack as opack

# Acceptance bar for the attention outputs: bf16 out within 1e-2 absolute +
# 1e-2 relative of the fp64 oracle, fp32 lse within 1e-3.
OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def device_cache(nvmla, w, dev, include_new=True):
    """Cache filled on the GPU by nvfp4_mla_pack with the workload's rows."""
    cache = torch.zeros((w.num_pages, 64, 352), dtype=torch.uint8, device=dev)
    if include_new:
        lat, rope, slots = w.all_written()
    else:
        lat, rope, slots = w.hist_latent, w.hist_rope, w.hist_slots
    if lat.shape[0]:
        nvmla.nvfp4_mla_pack(lat.to(dev), rope.to(dev), slots.to(dev), cache)
    return cache


def oracle_cache(w, tokens=None):
    """Cache packed by the oracle: every written row, or only the rows the
    listed tokens select (the oracle decode reads no others)."""
    lat, rope, slots = w.all_written()
    slots_np = slots.numpy().astype(np.int64)
    if tokens is not None:
        need = set()
        bt = w.block_table.numpy()
        L = w.seq_lens.numpy()
        for t in tokens:
            b = int(w.q_seq_idx[t])
            p = w.topk_idx[t].numpy().astype(np.int64)
            p = p[(p >= 0) & (p < L[b])]
            need.update((bt[b, p // 64].astype(np.int64) * 64 + p % 64).tolist())
        keep = np.isin(slots_np, np.fromiter(need, dtype=np.int64))
        lat, rope, slots_np = lat[keep], rope[keep], slots_np[keep]
    cache = np.zeros((w.num_pages, 64, 352), dtype=np.uint8)
    opack.pack_into_cache(lat.double().numpy(), rope.double().numpy(), slots_np, cache)
    return cache


def oracle_decode(w, cache_np, tokens=None, topk_idx=None):
    topk = w.topk_idx if topk_idx is None else topk_idx
    return oatt.sparse_mla_decode(w.q_latent, w.q_rope, cache_np, w.block_table, topk, w.sm_scale,
                                  w.q_seq_idx, w.seq_lens, tokens=tokens)


def device_inputs(w, dev):
    return dict(q_latent=w.q_latent.to(dev), q_rope=w.q_rope.to(dev), block_table=w.block_table.to(dev),
                topk_idx=w.topk_idx.to(dev), q_seq_idx=w.q_seq_idx.to(dev), seq_lens=w.seq_lens.to(dev))


def assert_close(out, lse, ref_out, ref_lse, what=""):
    """out: bf16 tensor [T', H, 512]; lse: fp32 [T', H]; refs float64."""
    o = out.float().cpu().double().numpy()
    l = lse.float().cpu().double().numpy()
    err = np.abs(o - ref_out)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    bad = err > bound
    assert not bad.any(), (f"{what}: out mismatch at {int(bad.sum())} of {bad.size} elements, "
                           f"max err {err.max():.3e}, first at {np.argwhere(bad)[0].tolist()}")
    inf_ref = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), inf_ref), f"{what}: lse -inf pattern differs"
    lerr = np.abs(l[~inf_ref] - ref_lse[~inf_ref])
    assert lerr.size == 0 or lerr.max() <= LSE_ATOL, f"{what}: lse max err {lerr.max():.3e}"
    return float(err.max()), float(lerr.max()) if lerr.size else 0.0
