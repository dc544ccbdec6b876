"""The synthetic input recipe checked against what it is meant to produce:
shapes and dtypes, index ranges and distinctness, the padding fractions, the
clustered lists' split between recent and older positions, the page mapping
(every logical page of every sequence on its own physical page), the rows
written before the decode (exactly the selected ones, plus the packed chunk),
and determinism under a fixed seed. The batched and write+read workloads run
at reduced counts here; their code paths are the same at full size."""
import math

import numpy as np
import torch

from nvfp4_sparse_mla_gb300 import workloads as wl

PAGE = 64


def _selected_slots(w):
    bt, tk, qs = w.block_table.numpy(), w.topk_idx.numpy(), w.q_seq_idx.numpy()
    sel = tk >= 0
    seqs = np.broadcast_to(qs[:, None], tk.shape)[sel]
    pos = tk[sel]
    return bt[seqs, pos // PAGE] * PAGE + pos % PAGE


def _check_common(w):
    lens = w.seq_lens.numpy()
    bt = w.block_table.numpy()
    used = np.concatenate([bt[b, :math.ceil(int(n) / PAGE)] for b, n in enumerate(lens)])
    assert len(np.unique(used)) == len(used) == w.num_pages
    assert used.min() >= 0 and used.max() < w.num_pages
    tk, qs = w.topk_idx.numpy(), w.q_seq_idx.numpy()
    assert qs.min() >= 0 and qs.max() < w.num_seqs
    lim = lens[qs][:, None]
    assert ((tk == -1) | ((tk >= 0) & (tk < lim))).all()
    for row in tk:
        v = row[row >= 0]
        assert len(np.unique(v)) == len(v)
    written = np.sort(w.all_written()[2].numpy())
    want = np.union1d(np.unique(_selected_slots(w)), w.new_slots.numpy())
    assert np.array_equal(written, want)
    assert w.q_latent.dtype == torch.bfloat16 and w.q_rope.dtype == torch.bfloat16
    assert tuple(w.q_latent.shape) == (w.T, w.H, 512) and tuple(w.q_rope.shape) == (w.T, w.H, 64)
    assert w.hist_latent.shape[1] == 512 and w.hist_rope.shape[1] == 64
    assert abs(w.sm_scale - 1.0 / math.sqrt(192.0)) < 1e-12


def test_tiny():
    w = wl.tiny()
    _check_common(w)
    assert (w.T, w.H, w.topk, int(w.seq_lens[0])) == (1, 16, 256, 4096)
    assert (w.topk_idx >= 0).all()


def test_decode_point():
    w = wl.decode_point()
    _check_common(w)
    assert (w.T, w.H, w.topk, w.num_seqs) == (15, 64, 2048, 1)
    assert int(w.seq_lens[0]) == 200_000 and w.num_pages == 3125
    assert (w.topk_idx >= 0).all()
    # uniform over the context: every tenth of it holds about a tenth
    counts = np.histogram(w.topk_idx.numpy(), bins=10, range=(0, 200_000))[0]
    assert counts.min() > 0.08 * w.topk_idx.numel()


def test_padded_fractions():
    w = wl.padded()
    _check_common(w)
    assert (w.T, w.topk, int(w.seq_lens[0])) == (35, 2048, 32_768)
    frac = (w.topk_idx == -1).float().mean(dim=1).numpy()
    assert frac.min() >= 0.0 and frac.max() <= 0.6 + 1.0 / 2048
    assert frac.max() > 0.3  # the fractions spread over U[0, 0.6]


def test_batched_lists_are_clustered():
    w = wl.batched(num_seqs=6)
    _check_common(w)
    lens = w.seq_lens.numpy()
    assert w.num_seqs == 6 and lens.min() >= 32_768 and lens.max() <= 140_000
    per = np.bincount(w.q_seq_idx.numpy(), minlength=6)
    assert per.min() >= 1 and per.max() <= 4
    tk, qs = w.topk_idx.numpy(), w.q_seq_idx.numpy()
    recent = (tk >= (lens[qs] - 6144)[:, None]).sum(axis=1)
    assert (recent == 1024).all()  # half the slots in the last 6K positions


def test_write_read_chunk_and_lists():
    w = wl.write_read(T=8)
    _check_common(w)
    assert w.T == 8 and int(w.seq_lens[0]) == 140_000
    # the packed chunk is the last 6,144 positions of the sequence
    bt = w.block_table.numpy()
    pos = np.arange(140_000 - 6144, 140_000)
    assert np.array_equal(np.sort(w.new_slots.numpy()), np.sort(bt[0, pos // PAGE] * PAGE + pos % PAGE))
    assert (w.topk_idx.numpy() >= 140_000 - 6144).sum(axis=1).tolist() == [1024] * 8
    # about 1% of the chunk's latent values are the x20 outliers
    big = (w.new_latent.float().abs() > 8.0).float().mean().item()
    assert 0.002 < big < 0.03


def test_fixed_seed_is_deterministic():
    a, b = wl.decode_point(T=3), wl.decode_point(T=3)
    for f in ("q_latent", "q_rope", "topk_idx", "block_table", "hist_latent", "hist_slots"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    c = wl.decode_point(seed=2, T=3)
    assert not torch.equal(a.topk_idx, c.topk_idx)


def test_pack_chunk_slots_are_distinct():
    lat, rope, slots = wl.pack_chunk(7, 5000, 200)
    s = slots.numpy()
    assert len(np.unique(s)) == 5000 and s.min() >= 0 and s.max() < 200 * PAGE
    assert lat.shape == (5000, 512) and rope.shape == (5000, 64) and lat.dtype == torch.bfloat16
