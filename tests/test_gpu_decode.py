"""GPU parity of sparse_mla_decode against the fp64 oracle.

Bar: bf16 out within 1e-2 absolute + 1e-2 relative, fp32 lse within 1e-3;
-inf lse (no valid slot) and zero output exactly. Every kernel the library
ships (mma.sync with split-key partials; tcgen05 where the head count allows
it) is checked on every workload."""
import math

import numpy as np
import pytest
import torch

import parity
from oracle import attention as oatt
from nvfp4_sparse_mla_gb300 import workloads

pytestmark = pytest.mark.gpu

IMPLS = ["auto", "mma", "tcgen05"]


def _impl(lib, name):
    return {"auto": None, "mma": lib.IMPL_MMA, "tcgen05": lib.IMPL_TCGEN05}[name]


def _skip_unsupported(impl, H):
    if impl == "tcgen05" and H % 64 != 0:
        pytest.skip("the tcgen05 kernel covers head counts that are multiples of 64")


@pytest.fixture(scope="module")
def tiny_setup(lib, cuda):
    w = workloads.tiny()
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    assert np.array_equal(cache.cpu().numpy(), ref_cache), "GPU pack differs from the oracle pack"
    return w, cache, ref_cache


def run(lib, w, cache, dev, impl=None, num_splits=None, **over):
    d = parity.device_inputs(w, dev)
    d.update(over)
    return lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"], w.sm_scale,
                                 q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"], impl=impl,
                                 num_splits=num_splits)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("splits", [None, 1, 3, 4])
def test_tiny(lib, cuda, tiny_setup, impl, splits):
    w, cache, ref_cache = tiny_setup
    _skip_unsupported(impl, w.H)
    ro, rl, _ = parity.oracle_decode(w, ref_cache)
    out, lse = run(lib, w, cache, cuda, impl=_impl(lib, impl), num_splits=splits)
    parity.assert_close(out, lse, ro, rl, f"tiny/{impl}/{splits}")


@pytest.mark.parametrize("name", ["decode_point", "padded"])
@pytest.mark.parametrize("impl", IMPLS)
def test_full_size_all_tokens(lib, cuda, name, impl):
    """The pages' decode point (15 tokens x top-2048, 200K context) and the
    padded-list workload (35 tokens, up to 60% empty slots), every output
    element."""
    w = workloads.make(name)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
    ro, rl, bad = parity.oracle_decode(w, ref_cache)
    assert bad == 0
    out, lse = run(lib, w, cache, cuda, impl=_impl(lib, impl))
    parity.assert_close(out, lse, ro, rl, f"{name}/{impl}")


@pytest.mark.parametrize("name,ntok", [("batched", 24), ("write_read", 16)])
@pytest.mark.parametrize("impl", IMPLS)
def test_full_size_sampled(lib, cuda, name, ntok, impl):
    """Batched decode (~160 tokens over 64 sequences) and the write+read
    workload (128 tokens): the whole call runs, sampled tokens are checked
    element by element."""
    w = workloads.make(name)
    cache = parity.device_cache(lib, w, cuda)
    rng = np.random.default_rng(0)
    toks = sorted(rng.choice(w.T, size=min(ntok, w.T), replace=False).tolist())
    ref_cache = parity.oracle_cache(w, tokens=toks)
    ro, rl, _ = parity.oracle_decode(w, ref_cache, tokens=toks)
    out, lse = run(lib, w, cache, cuda, impl=_impl(lib, impl))
    parity.assert_close(out[toks], lse[toks], ro, rl, f"{name}/{impl}")
    assert torch.isfinite(lse).all()


def _small(seed, T=3, H=64, ctx=1000, topk=300, pad=0.2):
    """A small multi-tile problem with a ragged tail (topk not a multiple of
    the tile) built from the shared generator's pieces."""
    rng = np.random.default_rng(seed)
    w = workloads.padded(seed=seed, T=T, H=H, ctx=ctx, topk=topk, max_pad_frac=pad)
    return w


@pytest.mark.parametrize("H", [16, 32, 48, 64, 128])
@pytest.mark.parametrize("topk", [1, 17, 64, 100, 300])
@pytest.mark.parametrize("impl", IMPLS)
def test_shapes(lib, cuda, H, topk, impl):
    _skip_unsupported(impl, H)
    w = workloads.padded(seed=100 + H + topk, T=3, H=H, ctx=700, topk=topk, max_pad_frac=0.3)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    ro, rl, _ = parity.oracle_decode(w, ref_cache)
    out, lse = run(lib, w, cache, cuda, impl=_impl(lib, impl))
    parity.assert_close(out, lse, ro, rl, f"H{H}/k{topk}/{impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_all_padding(lib, cuda, tiny_setup, impl):
    w, cache, _ = tiny_setup
    _skip_unsupported(impl, w.H)
    pad = torch.full_like(w.topk_idx, -1).to(cuda)
    out, lse = run(lib, w, cache, cuda, impl=_impl(lib, impl), topk_idx=pad)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("impl", IMPLS)
def test_padding_is_invisible(lib, cuda, impl):
    """Appending and interleaving -1 slots changes nothing (beyond fp32
    summation order)."""
    w = workloads.padded(seed=7, T=4, H=64, ctx=2000, topk=256, max_pad_frac=0.0)
    cache = parity.device_cache(lib, w, cuda)
    out, lse = run(lib, w, cache, cuda, impl=_impl(lib, impl))
    t = w.topk_idx
    padded = torch.cat([t, torch.full((t.shape[0], 200), -1, dtype=torch.int32)], 1)
    padded = padded[:, torch.randperm(padded.shape[1], generator=torch.Generator().manual_seed(0))]
    out2, lse2 = run(lib, w, cache, cuda, impl=_impl(lib, impl), topk_idx=padded.contiguous().to(cuda))
    assert torch.allclose(out.float(), out2.float(), atol=2e-3, rtol=1e-2)
    assert torch.allclose(lse, lse2, atol=1e-4)


@pytest.mark.parametrize("impl", IMPLS)
def test_bad_indices_masked_and_counted(lib, cuda, impl):
    w = workloads.padded(seed=8, T=2, H=64, ctx=1500, topk=128, max_pad_frac=0.0)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    t = w.topk_idx.clone()
    t[0, 5] = 1500          # == seq_len
    t[0, 9] = 10 ** 6       # far beyond
    t[1, 0] = -5            # negative but not -1
    t[1, 1] = -1            # padding: not an error
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    d = parity.device_inputs(w, cuda)
    out, lse = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], t.to(cuda), w.sm_scale,
                                     q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"], err_word=err,
                                     impl=_impl(lib, impl))
    ro, rl, bad = parity.oracle_decode(w, ref_cache, topk_idx=t)
    assert bad == 3
    parity.assert_close(out, lse, ro, rl, "bad indices")
    e = err.cpu().tolist()
    assert e[0] & 0x1 and e[1] == 3


@pytest.mark.parametrize("impl", IMPLS)
def test_bad_sequence_index_masks_the_token(lib, cuda, impl):
    """A query token whose sequence index has no block-table row reads
    nothing (out 0, lse -inf) and every entry of its list other than -1 is
    counted; the other tokens of the call are unaffected."""
    w = workloads.padded(seed=10, T=3, H=64, ctx=1200, topk=160, max_pad_frac=0.2)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    qs = w.q_seq_idx.clone()
    qs[1] = 5  # the workload has one sequence
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    d = parity.device_inputs(w, cuda)
    out, lse = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"], w.sm_scale,
                                     q_seq_idx=qs.to(cuda), seq_lens=d["seq_lens"], err_word=err,
                                     impl=_impl(lib, impl))
    ro, rl, bad = oatt.sparse_mla_decode(w.q_latent, w.q_rope, ref_cache, w.block_table, w.topk_idx, w.sm_scale,
                                         qs, w.seq_lens)
    assert bad == int((w.topk_idx[1] != -1).sum())
    parity.assert_close(out, lse, ro, rl, "bad sequence index")
    e = err.cpu().tolist()
    assert e[0] & 0x1 and e[1] == bad


@pytest.mark.parametrize("impl", IMPLS)
def test_duplicates_and_null_optionals(lib, cuda, impl):
    """Duplicated positions count once per slot; q_seq_idx / seq_lens may be
    omitted for a single sequence."""
    w = workloads.padded(seed=9, T=2, H=64, ctx=900, topk=200, max_pad_frac=0.0)
    t = w.topk_idx.clone()
    t[:, 100:] = t[:, :100]
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    d = parity.device_inputs(w, cuda)
    out, lse = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], t.to(cuda), w.sm_scale,
                                     impl=_impl(lib, impl))
    ro, rl, _ = parity.oracle_decode(w, ref_cache, topk_idx=t)
    parity.assert_close(out, lse, ro, rl, "duplicates")


def test_zero_tokens_is_noop(lib, cuda, tiny_setup):
    w, cache, _ = tiny_setup
    d = parity.device_inputs(w, cuda)
    out, lse = lib.sparse_mla_decode(d["q_latent"][:0], d["q_rope"][:0], cache, d["block_table"],
                                     d["topk_idx"][:0], w.sm_scale)
    assert out.shape == (0, 16, 512)


def test_small_workspace_falls_back(lib, cuda, tiny_setup):
    """A workspace too small for the default split count gives the same
    result with fewer splits."""
    w, cache, ref_cache = tiny_setup
    ro, rl, _ = parity.oracle_decode(w, ref_cache)
    d = parity.device_inputs(w, cuda)
    ws = torch.empty(16, dtype=torch.uint8, device=cuda)
    out, lse = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"], w.sm_scale,
                                     workspace=ws, impl=lib.IMPL_MMA)
    parity.assert_close(out, lse, ro, rl, "fallback")


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8, 16])
def test_tcgen05_splits(lib, cuda, splits):
    """The tcgen05 kernel with explicit key splits (single CTA per token up to
    one CTA per 128-row tile), on the decode-point shape with fewer tokens."""
    w = workloads.decode_point(seed=11, T=3, ctx=50_000)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    ro, rl, _ = parity.oracle_decode(w, ref_cache)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    d = parity.device_inputs(w, cuda)
    try:
        out, lse = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"],
                                         w.sm_scale, q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"], err_word=err,
                                         impl=lib.IMPL_TCGEN05, num_splits=splits)
    except lib.NvmlaError as e:
        # more than 8 CTAs per cluster is a device option
        if splits > 8 and e.status == 2 and "cluster" in str(e):
            pytest.skip(str(e))
        raise
    parity.assert_close(out, lse, ro, rl, f"tcgen05 splits={splits}")
    assert err.cpu().tolist() == [0, 0]


def test_tcgen05_rejects_other_head_counts(lib, cuda, tiny_setup):
    w, cache, _ = tiny_setup
    d = parity.device_inputs(w, cuda)
    with pytest.raises(lib.NvmlaError):
        lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"], w.sm_scale,
                              impl=lib.IMPL_TCGEN05)


def test_large_score_range_rescales(lib, cuda):
    """Scores spread over a wide range (queries scaled x8) force the running
    maximum up across tiles, exercising the rescale of the accumulator."""
    w = workloads.decode_point(seed=12, T=2, ctx=20_000)
    w.q_latent = (w.q_latent.float() * 8).to(torch.bfloat16)
    w.q_rope = (w.q_rope.float() * 8).to(torch.bfloat16)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    ro, rl, _ = parity.oracle_decode(w, ref_cache)
    for impl in (lib.IMPL_MMA, lib.IMPL_TCGEN05):
        for splits in (1, 2):
            d = parity.device_inputs(w, cuda)
            out, lse = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"],
                                             w.sm_scale, q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"],
                                             impl=impl, num_splits=splits)
            parity.assert_close(out, lse, ro, rl, f"wide scores impl={impl} splits={splits}")


@pytest.mark.parametrize("splits", [1, 4])
def test_forced_wait_timeout_reports_and_recovers(lib, cuda, splits):
    """The tcgen05 kernel's bounded-wait abort path, made to run by the test
    hook that has the MMA thread's wait for P^T give up at once: the call
    completes (every CTA drains its MMAs, frees TMEM and meets the cluster
    barriers), err_word carries NVMLA_ERRW_WAIT_TIMEOUT, and the next normal
    call on the same stream matches the oracle."""
    w = workloads.decode_point(seed=13, T=3, ctx=20_000)
    cache = parity.device_cache(lib, w, cuda)
    ref_cache = parity.oracle_cache(w)
    ro, rl, _ = parity.oracle_decode(w, ref_cache)
    d = parity.device_inputs(w, cuda)
    err = torch.zeros(2, dtype=torch.int32, device=cuda)
    lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"], w.sm_scale,
                          q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"], err_word=err, impl=lib.IMPL_TCGEN05,
                          num_splits=splits, debug_flags=lib.DEBUG_FORCE_WAIT_TIMEOUT)
    torch.cuda.synchronize()
    flags, count = err.cpu().tolist()
    assert flags == 8 and count >= 1, (flags, count)  # NVMLA_ERRW_WAIT_TIMEOUT only
    err.zero_()
    out, lse = lib.sparse_mla_decode(d["q_latent"], d["q_rope"], cache, d["block_table"], d["topk_idx"], w.sm_scale,
                                     q_seq_idx=d["q_seq_idx"], seq_lens=d["seq_lens"], err_word=err,
                                     impl=lib.IMPL_TCGEN05, num_splits=splits)
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    parity.assert_close(out, lse, ro, rl, f"after a forced timeout, splits={splits}")
