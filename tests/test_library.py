"""Host-side checks of the C-ABI library (no GPU needed): it builds, loads,
exports every function include/nvmla.h declares, and rejects bad arguments
with an error status before launching anything."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "nvmla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ["nvfp4_mla_pack", "sparse_mla_decode", "sparse_mla_decode_workspace_size",
              "nvfp4_stage_dequant_fp8", "sparse_mla_decode_fp8rows", "nvmla_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.library_path())
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_binding_uses_the_library(lib):
    assert lib.load().nvmla_version() >= 100
    assert os.path.dirname(lib.library_path()) == os.path.join(ROOT, "nvfp4_sparse_mla_gb300")


def _raw(lib):
    return lib.load()


def test_decode_rejects_bad_arguments(lib):
    L = _raw(lib)
    P = ctypes.c_void_p
    ok = P(0x10000)  # never dereferenced: validation fails first

    def call(**kw):
        a = dict(ql=ok, qr=ok, cache=ok, pages=10, bt=ok, nseq=1, maxp=4, topk_idx=ok, topk=2048, qs=None, sl=None,
                 T=15, H=64, scale=0.1, out=ok, lse=ok, ws=None, wsb=0, err=None, stream=None)
        a.update(kw)
        return L.sparse_mla_decode(*a.values())

    assert call(ql=None) == 1
    assert call(out=None) == 1
    assert call(cache=P(0x10008)) == 1          # misaligned cache
    assert call(H=40) == 2                      # not a multiple of 16
    assert call(H=144) == 2
    assert call(topk=0) == 2 and call(topk=4096) == 2
    assert call(T=-1) == 1
    assert call(pages=0) == 1
    assert call(scale=float("nan")) == 1
    assert call(T=0) == 0                       # no-op, nothing touched
    assert b"topk" in L.nvmla_last_error() or True


def test_pack_rejects_bad_arguments(lib):
    L = _raw(lib)
    P = ctypes.c_void_p
    ok = P(0x10000)

    def call(**kw):
        a = dict(lat=ok, ls=512, rope=ok, rs=64, slots=ok, n=10, cache=ok, pages=1, err=None, stream=None)
        a.update(kw)
        return L.nvfp4_mla_pack(*a.values())

    assert call(lat=None) == 1
    assert call(ls=500) == 1
    assert call(ls=516) == 1                    # not a multiple of 8
    assert call(rope=P(0x10002)) == 1
    assert call(cache=P(0x10004)) == 1
    assert call(n=-1) == 1
    assert call(n=0) == 0
    assert b"" != L.nvmla_last_error()


def test_staged_rejects_bad_arguments(lib):
    L = _raw(lib)
    P = ctypes.c_void_p
    ok = P(0x10000)
    assert L.nvfp4_stage_dequant_fp8(ok, 4, ok, 1, 4, ok, 2048, None, None, 3, None, ok, None, None) == 1
    assert L.nvfp4_stage_dequant_fp8(ok, 4, ok, 1, 4, ok, 0, None, None, 3, ok, ok, None, None) == 2
    assert L.sparse_mla_decode_fp8rows(ok, ok, None, ok, 2048, 3, 64, 0.1, ok, ok, None, 0, None, None, None) == 1


def test_python_binding_checks_dtypes(lib):
    q = torch.zeros((1, 16, 512), dtype=torch.float32)
    with pytest.raises(ValueError):
        lib.sparse_mla_decode(q, q, torch.zeros((1, 64, 352), dtype=torch.uint8),
                              torch.zeros((1, 1), dtype=torch.int32), torch.zeros((1, 4), dtype=torch.int32), 0.1)


def test_workspace_size_is_host_only(lib):
    assert lib.sparse_mla_decode_workspace_size(15, 64, 2048, impl=lib.IMPL_MMA, num_splits=1) == 0
    n = lib.sparse_mla_decode_workspace_size(15, 64, 2048, impl=lib.IMPL_MMA, num_splits=8)
    assert n == 15 * 8 * 64 * 514 * 4


@pytest.mark.skipif(torch.cuda.is_available(), reason="on a GPU the device's own cluster occupancy decides")
def test_default_split_counts_follow_the_wave_cost_model(lib):
    # Without a device the library assumes 152 SMs holding 152 / S clusters
    # of S CTAs (S <= 8). Cost of S: waves * (19 + 5 * ceil(16 / S)) us, the
    # cheapest S, then the fewest splits with the same tiles per CTA. The
    # kernel takes no workspace: its partials stay in shared memory.
    def splits(T, H=64):
        assert lib.sparse_mla_decode_workspace_size(T, H, 2048, impl=lib.IMPL_TCGEN05) == 0
        return lib.sparse_mla_decode_splits(T, H, 2048, impl=lib.IMPL_TCGEN05)

    assert splits(1) == 8      # one wave: 19 + 10
    assert splits(15) == 8     # 15 clusters of 8 fit (19 resident)
    assert splits(24) == 6     # 6 -> 3 tiles a CTA in one wave (34) beats 8 in two (58)
    assert splits(35) == 4     # 38 clusters of 4 fit; 5 would need two waves
    assert splits(64) == 2     # 59 against 98 for 3 splits
    assert splits(128) == 1    # 99 against 118 for two waves of pairs
    assert splits(160) == 2    # three waves of pairs (177) beat two of single CTAs (198)
    assert splits(256) == 1    # 198 against 236
    assert splits(320) == 2    # 295 against 297
    assert splits(15, H=128) == 4  # 30 clusters: 5 splits of at most 4 tiles, reduced to 4


def test_short_names_are_the_calls(lib):
    assert lib.pack is lib.nvfp4_mla_pack and lib.decode is lib.sparse_mla_decode
    assert {"pack", "decode"} <= set(lib.__all__)


def test_layered_calls_reject_bad_layers(lib):
    L = _raw(lib)
    P = ctypes.c_void_p
    ok = P(0x10000)

    def dec(**kw):
        a = dict(ql=ok, qr=ok, cache=ok, blocks=10, layers=4, layer=1, bt=ok, nseq=1, maxp=4, topk_idx=ok, topk=2048,
                 qs=None, sl=None, T=15, H=64, scale=0.1, out=ok, lse=ok, ws=None, wsb=0, err=None, opts=None,
                 stream=None)
        a.update(kw)
        return L.sparse_mla_decode_layered(*a.values())

    def pk(**kw):
        a = dict(lat=ok, ls=512, rope=ok, rs=64, slots=ok, n=10, cache=ok, blocks=1, layers=4, layer=1, err=None,
                 stream=None)
        a.update(kw)
        return L.nvfp4_mla_pack_layered(*a.values())

    for call in (dec, pk):
        assert call(layer=4) == 1
        assert call(layer=-1) == 1
        assert call(layers=0, layer=0) == 1
        assert call(layers=5000, layer=0) == 1
        assert call(cache=P(0x10010)) == 1      # misaligned cache
        assert b"" != L.nvmla_last_error()
    assert dec(T=0) == 0 and pk(n=0) == 0       # no-ops, nothing touched


def test_topk_select_rejects_bad_arguments(lib):
    L = _raw(lib)
    P = ctypes.c_void_p
    ok = P(0x10000)
    assert L.nvmla_topk_select(ok, 100, 100, None, 3, 0, ok, None) == 2        # topk 0
    assert L.nvmla_topk_select(ok, 100, 100, None, 3, 4096, ok, None) == 2     # topk > 2048
    assert L.nvmla_topk_select(ok, 50, 100, None, 3, 2048, ok, None) == 1      # stride < ncols
    assert L.nvmla_topk_select(None, 100, 100, None, 3, 2048, ok, None) == 1
    assert L.nvmla_topk_select(ok, 100, 100, None, 3, 2048, None, None) == 1
    assert L.nvmla_topk_select(P(0x10002), 100, 100, None, 3, 2048, ok, None) == 1
    assert L.nvmla_topk_select(ok, 100, 100, None, -1, 2048, ok, None) == 1
    assert L.nvmla_topk_select(ok, 100, 100, None, 0, 2048, ok, None) == 0     # no-op
    assert L.nvmla_topk_select(ok, 100, 100, None, 65536, 2048, ok, None) == 2  # T beyond the grid
    big = (1 << 29) + 1
    assert L.nvmla_topk_select(ok, big, big, None, 3, 2048, ok, None) == 2     # row too long


def test_decode_rejects_too_many_tokens(lib):
    L = _raw(lib)
    ok = ctypes.c_void_p(0x10000)
    args = [ok, ok, ok, 10, ok, 1, 4, ok, 2048, None, None, 65536, 64, 0.1, ok, ok, None, 0, None, None]
    assert L.sparse_mla_decode(*args) == 2


def test_fp8_cache_calls_reject_bad_arguments(lib):
    L = _raw(lib)
    P = ctypes.c_void_p
    ok = P(0x10000)
    assert L.fp8_mla_pack(None, 512, ok, 64, ok, 10, ok, 1, None, None) == 1
    assert L.fp8_mla_pack(ok, 512, ok, 64, ok, 10, P(0x10008), 1, None, None) == 1
    assert L.fp8_mla_pack(ok, 512, ok, 64, ok, 0, ok, 1, None, None) == 0
    args = [ok, ok, ok, 10, ok, 1, 4, ok, 2048, None, None, 15, 32, 0.1, ok, ok, None, 0, None, None, None]
    assert L.sparse_mla_decode_fp8cache(*args) == 2            # H = 32: not on the tcgen05 kernel
    args[12] = 64
    args[2] = P(0x10008)
    assert L.sparse_mla_decode_fp8cache(*args) == 1            # misaligned cache


_CONCURRENT_QUERIES = r"""
import ctypes, sys, threading
import nvfp4_sparse_mla_gb300 as nvmla
lib = nvmla.load()
shapes = [(T, H, k) for T in (1, 7, 15, 24, 35, 64, 128, 320) for H in (16, 48, 64, 128) for k in (512, 2048)]
def run():
    return [(nvmla.sparse_mla_decode_workspace_size(T, H, k), nvmla.sparse_mla_decode_splits(T, H, k))
            for (T, H, k) in shapes]
start = threading.Barrier(8)
results = [None] * 8
def worker(i):
    start.wait()
    results[i] = [run() for _ in range(20)]
threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
for t in threads: t.start()
for t in threads: t.join()
ref = run()
bad = sum(r != ref for per in results for r in per)
print("shapes", len(shapes), "mismatches", bad)
sys.exit(1 if bad else 0)
"""


def test_size_queries_from_eight_threads_at_first_use(lib):
    """A fresh process whose first calls into the library come from eight
    threads at once (ctypes drops the GIL): each thread's workspace sizes and
    split counts equal the ones a single thread sees afterwards. On a GPU this
    races the per-device launch set-up; without one, the host-only model."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CONCURRENT_QUERIES], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout


def test_in_tree_library_is_the_default_build(lib):
    """The library the package loads has no debug checks compiled in (the
    bounds-checked build is a separate variant the GPU tests build)."""
    assert lib.library_path().endswith("libnvmla.so")
    assert lib.build_flags() == 0
