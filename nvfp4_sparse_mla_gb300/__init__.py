"""NVFP4 sparse-MLA decode for GB300: Python binding of the C-ABI library.

The binding only marshals arguments: it checks dtypes and shapes, takes
device pointers and the current CUDA stream from torch tensors, allocates
missing outputs with torch, and calls ``libnvmla.so``. Every step of the
computation runs in the library's CUDA kernels; there is no other code path.
If the library has not been built (``python -m nvfp4_sparse_mla_gb300._build``)
every call raises.

Calls (same names as the C ABI, see include/nvmla.h):

* ``nvfp4_mla_pack(latent, rope, slot_mapping, cache)`` (also ``pack``)
* ``sparse_mla_decode(q_latent, q_rope, cache, block_table, topk_idx, sm_scale, ...)`` (also ``decode``)
* ``sparse_mla_decode_noalloc(q_latent, q_rope, cache, block_table, topk_idx, sm_scale, out, lse, ...)``
  (the same decode with the library's own split scratch; allocates nothing)
* ``nvfp4_mla_pack_layered(latent, rope, slot_mapping, cache, layer)`` and
  ``sparse_mla_decode_layered(q_latent, q_rope, cache, layer, block_table, topk_idx, sm_scale, ...)``
  (one layer of a block-major multi-layer cache [num_blocks, num_layers, 64, 352])
* ``fp8_mla_pack(latent, rope, slot_mapping, cache)`` and
  ``sparse_mla_decode_fp8cache(q_latent, q_rope, cache, block_table, topk_idx, sm_scale, ...)``
  (the 576-byte FP8 cache the NVFP4 format is measured against)
* ``nvmla_topk_select(scores, topk, lengths=None)`` (the -1 padded top-k
  lists the decode consumes, from given scores)
* ``nvfp4_stage_dequant_fp8(cache, block_table, topk_idx, ...)`` and
  ``sparse_mla_decode_fp8rows(q_latent, q_rope, fp8_rows, row_idx, sm_scale, ...)``
  (the staged baseline)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "NvmlaError", "nvfp4_mla_pack", "sparse_mla_decode", "sparse_mla_decode_workspace_size", "sparse_mla_decode_fp8rows_workspace_size", "launch_count",
    "nvfp4_stage_dequant_fp8", "sparse_mla_decode_fp8rows", "library_path", "load",
    "sparse_mla_decode_noalloc", "sparse_mla_decode_noalloc_max_scratch",
    "nvfp4_mla_pack_layered", "sparse_mla_decode_layered", "nvmla_topk_select",
    "fp8_mla_pack", "sparse_mla_decode_fp8cache",
    "IMPL_AUTO", "IMPL_MMA", "IMPL_TCGEN05", "ROW_BYTES", "FP8_ROW_BYTES", "PAGE_TOKENS",
    "pack", "decode",
]

ROW_BYTES = 352
FP8_ROW_BYTES = 576
PAGE_TOKENS = 64
IMPL_AUTO, IMPL_MMA, IMPL_TCGEN05 = 0, 1, 2
DEBUG_FORCE_WAIT_TIMEOUT = 0x1  # NVMLA_DEBUG_FORCE_WAIT_TIMEOUT (a test hook)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libnvmla.so"
_lib = None


class NvmlaError(RuntimeError):
    """A library call returned an error status."""

    def __init__(self, status: int, name: str, message: str):
        super().__init__(f"{name}: {message}")
        self.status = status
        self.name = name


class _Options(ctypes.Structure):
    _fields_ = [("impl", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("debug_flags", ctypes.c_int32)]


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load():
    """Load libnvmla.so (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m nvfp4_sparse_mla_gb300._build`")
    lib = ctypes.CDLL(path)
    P, I32, I64, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    OPT = ctypes.POINTER(_Options)
    sig = {
        "nvfp4_mla_pack": (I32, [P, I64, P, I64, P, I64, P, I64, P, P]),
        "sparse_mla_decode": (I32, [P, P, P, I64, P, I32, I32, P, I32, P, P, I32, I32, F, P, P, P, SZ, P, P]),
        "sparse_mla_decode_ex": (I32, [P, P, P, I64, P, I32, I32, P, I32, P, P, I32, I32, F, P, P, P, SZ, P, OPT, P]),
        "nvfp4_mla_pack_layered": (I32, [P, I64, P, I64, P, I64, P, I64, I32, I32, P, P]),
        "sparse_mla_decode_layered": (I32, [P, P, P, I64, I32, I32, P, I32, I32, P, I32, P, P, I32, I32, F, P, P, P, SZ,
                                            P, OPT, P]),
        "sparse_mla_decode_workspace_size": (SZ, [I32, I32, I32]),
        "sparse_mla_decode_workspace_size_ex": (SZ, [I32, I32, I32, OPT]),
        "sparse_mla_decode_splits": (I32, [I32, I32, I32, OPT]),
        "sparse_mla_decode_noalloc": (I32, [P, P, P, I64, P, I32, I32, P, I32, P, P, I32, I32, F, P, P, P, P]),
        "sparse_mla_decode_noalloc_max_scratch": (SZ, []),
        "nvfp4_stage_dequant_fp8": (I32, [P, I64, P, I32, I32, P, I32, P, P, I32, P, P, P, P]),
        "sparse_mla_decode_fp8rows": (I32, [P, P, P, P, I32, I32, I32, F, P, P, P, SZ, P, OPT, P]),
        "sparse_mla_decode_fp8rows_workspace_size": (SZ, [I32, I32, I32, OPT]),
        "nvmla_topk_select": (I32, [P, I64, I32, P, I32, I32, P, P]),
        "fp8_mla_pack": (I32, [P, I64, P, I64, P, I64, P, I64, P, P]),
        "sparse_mla_decode_fp8cache": (I32, [P, P, P, I64, P, I32, I32, P, I32, P, P, I32, I32, F, P, P, P, SZ, P, OPT,
                                             P]),
        "nvmla_status_string": (ctypes.c_char_p, [I32]),
        "nvmla_last_error": (ctypes.c_char_p, []),
        "nvmla_version": (I32, []),
        "nvmla_launch_count": (ctypes.c_uint64, []),
        "nvmla_build_flags": (I32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def launch_count() -> int:
    """Kernels the library has launched so far in this process."""
    return int(load().nvmla_launch_count())


BUILD_DEBUG_BOUNDS = 0x1


def build_flags() -> int:
    """How the loaded library was compiled (BUILD_DEBUG_BOUNDS: the
    bounds-checked debug build)."""
    return int(load().nvmla_build_flags())


def _check(status: int):
    if status != 0:
        lib = load()
        raise NvmlaError(status, lib.nvmla_status_string(status).decode(), lib.nvmla_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream):
    if stream is not None:
        return ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)
    if t.is_cuda:
        return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)
    return None


def _need(t, name, dtype, dims=None, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got shape {tuple(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _opts(impl, num_splits, debug_flags=None):
    if impl is None and num_splits is None and not debug_flags:
        return None
    return ctypes.pointer(_Options(int(impl or 0), int(num_splits or 0), int(debug_flags or 0)))


def nvfp4_mla_pack(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor, cache: torch.Tensor,
                   err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Quantise latent [N,512] / rope [N,64] (bf16) into cache rows
    [num_pages, 64, 352] (uint8) at slot_mapping [N] (int32). Returns cache."""
    _need(latent, "latent", torch.bfloat16, 2, contiguous=False)
    _need(rope, "rope", torch.bfloat16, 2, contiguous=False)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(cache, "cache", torch.uint8, 3)
    if latent.shape[1] != 512 or rope.shape[1] != 64 or latent.stride(1) != 1 or rope.stride(1) != 1:
        raise ValueError("latent must be [N, 512] and rope [N, 64] with unit inner stride")
    n = latent.shape[0]
    if rope.shape[0] != n or slot_mapping.shape[0] != n:
        raise ValueError("latent, rope and slot_mapping must have the same number of tokens")
    if cache.shape[1:] != (PAGE_TOKENS, ROW_BYTES):
        raise ValueError("cache must be [num_pages, 64, 352]")
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, 1)
    lib = load()
    # the stride of a single-row tensor is meaningless (torch may report 0)
    ls = latent.stride(0) if n > 1 else 512
    rs = rope.stride(0) if n > 1 else 64
    _check(lib.nvfp4_mla_pack(_ptr(latent), ls, _ptr(rope), rs, _ptr(slot_mapping), n,
                              _ptr(cache), cache.shape[0], _ptr(err_word), _stream(cache, stream)))
    return cache


def _layered_cache(cache: torch.Tensor, layer: int):
    _need(cache, "cache", torch.uint8, 4)
    if cache.shape[2:] != (PAGE_TOKENS, ROW_BYTES):
        raise ValueError("cache must be [num_blocks, num_layers, 64, 352]")
    if not 0 <= int(layer) < cache.shape[1]:
        raise ValueError(f"layer {layer} outside [0, {cache.shape[1]})")


def nvfp4_mla_pack_layered(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor, cache: torch.Tensor,
                           layer: int, err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """nvfp4_mla_pack into layer `layer` of a block-major multi-layer cache
    [num_blocks, num_layers, 64, 352] (uint8); slots are block * 64 + token
    as for a one-layer cache. Returns cache."""
    _need(latent, "latent", torch.bfloat16, 2, contiguous=False)
    _need(rope, "rope", torch.bfloat16, 2, contiguous=False)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _layered_cache(cache, layer)
    if latent.shape[1] != 512 or rope.shape[1] != 64 or latent.stride(1) != 1 or rope.stride(1) != 1:
        raise ValueError("latent must be [N, 512] and rope [N, 64] with unit inner stride")
    n = latent.shape[0]
    if rope.shape[0] != n or slot_mapping.shape[0] != n:
        raise ValueError("latent, rope and slot_mapping must have the same number of tokens")
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, 1)
    lib = load()
    ls = latent.stride(0) if n > 1 else 512
    rs = rope.stride(0) if n > 1 else 64
    _check(lib.nvfp4_mla_pack_layered(_ptr(latent), ls, _ptr(rope), rs, _ptr(slot_mapping), n, _ptr(cache),
                                      cache.shape[0], cache.shape[1], int(layer), _ptr(err_word),
                                      _stream(cache, stream)))
    return cache


def sparse_mla_decode_layered(q_latent: torch.Tensor, q_rope: torch.Tensor, cache: torch.Tensor, layer: int,
                              block_table: torch.Tensor, topk_idx: torch.Tensor, sm_scale: float,
                              out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                              q_seq_idx: Optional[torch.Tensor] = None, seq_lens: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None, err_word: Optional[torch.Tensor] = None,
                              impl=None, num_splits=None, stream=None):
    """sparse_mla_decode over layer `layer` of a block-major multi-layer cache
    [num_blocks, num_layers, 64, 352]. Returns (out, lse)."""
    _need(q_latent, "q_latent", torch.bfloat16, 3)
    _need(q_rope, "q_rope", torch.bfloat16, 3)
    _layered_cache(cache, layer)
    _need(block_table, "block_table", torch.int32, 2)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    T, H, dl = q_latent.shape
    if dl != 512 or tuple(q_rope.shape) != (T, H, 64):
        raise ValueError("q_latent must be [T, H, 512] and q_rope [T, H, 64]")
    if topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, topk]")
    if q_seq_idx is not None:
        _need(q_seq_idx, "q_seq_idx", torch.int32, 1)
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, 1)
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q_latent.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q_latent.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    topk = topk_idx.shape[1]
    opts = _opts(impl, num_splits)
    lib = load()
    if workspace is None:
        nbytes = int(lib.sparse_mla_decode_workspace_size_ex(T, H, topk, opts))
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q_latent.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sparse_mla_decode_layered(_ptr(q_latent), _ptr(q_rope), _ptr(cache), cache.shape[0], cache.shape[1],
                                         int(layer), _ptr(block_table), block_table.shape[0], block_table.shape[1],
                                         _ptr(topk_idx), topk, _ptr(q_seq_idx), _ptr(seq_lens), T, H,
                                         float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                         _ptr(err_word), opts, _stream(q_latent, stream)))
    return out, lse


def fp8_mla_pack(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor, cache: torch.Tensor,
                 err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Write latent [N,512] / rope [N,64] (bf16) as 576-byte E4M3 rows into
    cache [num_pages, 64, 576] (uint8) at slot_mapping [N]. Returns cache."""
    _need(latent, "latent", torch.bfloat16, 2, contiguous=False)
    _need(rope, "rope", torch.bfloat16, 2, contiguous=False)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(cache, "cache", torch.uint8, 3)
    if latent.shape[1] != 512 or rope.shape[1] != 64 or latent.stride(1) != 1 or rope.stride(1) != 1:
        raise ValueError("latent must be [N, 512] and rope [N, 64] with unit inner stride")
    n = latent.shape[0]
    if rope.shape[0] != n or slot_mapping.shape[0] != n:
        raise ValueError("latent, rope and slot_mapping must have the same number of tokens")
    if cache.shape[1:] != (PAGE_TOKENS, FP8_ROW_BYTES):
        raise ValueError("cache must be [num_pages, 64, 576]")
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, 1)
    lib = load()
    ls = latent.stride(0) if n > 1 else 512
    rs = rope.stride(0) if n > 1 else 64
    _check(lib.fp8_mla_pack(_ptr(latent), ls, _ptr(rope), rs, _ptr(slot_mapping), n, _ptr(cache), cache.shape[0],
                            _ptr(err_word), _stream(cache, stream)))
    return cache


def sparse_mla_decode_fp8cache(q_latent: torch.Tensor, q_rope: torch.Tensor, cache: torch.Tensor,
                               block_table: torch.Tensor, topk_idx: torch.Tensor, sm_scale: float,
                               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                               q_seq_idx: Optional[torch.Tensor] = None, seq_lens: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None, err_word: Optional[torch.Tensor] = None,
                               num_splits=None, stream=None):
    """Sparse MLA decode over the FP8 cache [num_pages, 64, 576] (tcgen05
    kernel; H a multiple of 64). Returns (out, lse)."""
    _need(q_latent, "q_latent", torch.bfloat16, 3)
    _need(q_rope, "q_rope", torch.bfloat16, 3)
    _need(cache, "cache", torch.uint8, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    T, H, dl = q_latent.shape
    if dl != 512 or tuple(q_rope.shape) != (T, H, 64):
        raise ValueError("q_latent must be [T, H, 512] and q_rope [T, H, 64]")
    if topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, topk]")
    if cache.shape[1:] != (PAGE_TOKENS, FP8_ROW_BYTES):
        raise ValueError("cache must be [num_pages, 64, 576]")
    if q_seq_idx is not None:
        _need(q_seq_idx, "q_seq_idx", torch.int32, 1)
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, 1)
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q_latent.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q_latent.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    topk = topk_idx.shape[1]
    opts = _opts(IMPL_TCGEN05, num_splits)
    lib = load()
    if workspace is None:
        nbytes = int(lib.sparse_mla_decode_workspace_size_ex(T, H, topk, opts))
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q_latent.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sparse_mla_decode_fp8cache(_ptr(q_latent), _ptr(q_rope), _ptr(cache), cache.shape[0],
                                          _ptr(block_table), block_table.shape[0], block_table.shape[1],
                                          _ptr(topk_idx), topk, _ptr(q_seq_idx), _ptr(seq_lens), T, H,
                                          float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                          _ptr(err_word), opts, _stream(q_latent, stream)))
    return out, lse


def nvmla_topk_select(scores: torch.Tensor, topk: int = 2048, lengths: Optional[torch.Tensor] = None,
                      out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Top-k positions by score per row of scores [T, ncols] (fp32, unit
    inner stride), the first lengths[t] columns of row t being candidates;
    returns int32 [T, topk]: chosen positions in increasing order, then -1."""
    _need(scores, "scores", torch.float32, 2, contiguous=False)
    if scores.shape[1] > 0 and scores.stride(1) != 1:
        raise ValueError("scores must have unit inner stride")
    T, ncols = scores.shape
    if lengths is not None:
        _need(lengths, "lengths", torch.int32, 1)
        if lengths.shape[0] != T:
            raise ValueError("lengths must be [T]")
    if out is None:
        out = torch.empty((T, topk), dtype=torch.int32, device=scores.device)
    _need(out, "out", torch.int32, 2)
    if tuple(out.shape) != (T, topk):
        raise ValueError("out must be [T, topk]")
    stride = scores.stride(0) if T > 1 else ncols
    lib = load()
    _check(lib.nvmla_topk_select(_ptr(scores), max(stride, ncols), ncols, _ptr(lengths), T, int(topk), _ptr(out),
                                 _stream(scores, stream)))
    return out


def sparse_mla_decode_workspace_size(T: int, H: int, topk: int, impl=None, num_splits=None) -> int:
    lib = load()
    return int(lib.sparse_mla_decode_workspace_size_ex(T, H, topk, _opts(impl, num_splits)))


def sparse_mla_decode_splits(T: int, H: int, topk: int, impl=None, num_splits=None) -> int:
    """Key splits per token the decode takes for (T, H, topk) on the current
    device (0 for a shape it rejects)."""
    lib = load()
    return int(lib.sparse_mla_decode_splits(T, H, topk, _opts(impl, num_splits)))


def sparse_mla_decode_fp8rows_workspace_size(T: int, H: int, topk: int, impl=None, num_splits=None) -> int:
    lib = load()
    return int(lib.sparse_mla_decode_fp8rows_workspace_size(T, H, topk, _opts(impl, num_splits)))


def sparse_mla_decode(q_latent: torch.Tensor, q_rope: torch.Tensor, cache: torch.Tensor, block_table: torch.Tensor,
                      topk_idx: torch.Tensor, sm_scale: float, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, q_seq_idx: Optional[torch.Tensor] = None,
                      seq_lens: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      err_word: Optional[torch.Tensor] = None, impl=None, num_splits=None, stream=None,
                      debug_flags=None):
    """Sparse MLA decode over the NVFP4 cache. Returns (out bf16 [T,H,512],
    lse fp32 [T,H]). debug_flags: the NVMLA_DEBUG_* test hooks (None in
    normal use)."""
    _need(q_latent, "q_latent", torch.bfloat16, 3)
    _need(q_rope, "q_rope", torch.bfloat16, 3)
    _need(cache, "cache", torch.uint8, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    T, H, dl = q_latent.shape
    if dl != 512 or tuple(q_rope.shape) != (T, H, 64):
        raise ValueError("q_latent must be [T, H, 512] and q_rope [T, H, 64]")
    if topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, topk]")
    if cache.shape[1:] != (PAGE_TOKENS, ROW_BYTES):
        raise ValueError("cache must be [num_pages, 64, 352]")
    if q_seq_idx is not None:
        _need(q_seq_idx, "q_seq_idx", torch.int32, 1)
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, 1)
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q_latent.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q_latent.device)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    topk = topk_idx.shape[1]
    opts = _opts(impl, num_splits, debug_flags)
    lib = load()
    if workspace is None:
        nbytes = int(lib.sparse_mla_decode_workspace_size_ex(T, H, topk, opts))
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q_latent.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sparse_mla_decode_ex(_ptr(q_latent), _ptr(q_rope), _ptr(cache), cache.shape[0], _ptr(block_table),
                                    block_table.shape[0], block_table.shape[1], _ptr(topk_idx), topk,
                                    _ptr(q_seq_idx), _ptr(seq_lens), T, H, float(sm_scale), _ptr(out), _ptr(lse),
                                    _ptr(workspace), ws_bytes, _ptr(err_word), opts, _stream(q_latent, stream)))
    return out, lse


def sparse_mla_decode_noalloc_max_scratch() -> int:
    """Bytes of split scratch the library holds per device for
    sparse_mla_decode_noalloc."""
    return int(load().sparse_mla_decode_noalloc_max_scratch())


def sparse_mla_decode_noalloc(q_latent: torch.Tensor, q_rope: torch.Tensor, cache: torch.Tensor,
                              block_table: torch.Tensor, topk_idx: torch.Tensor, sm_scale: float,
                              out: torch.Tensor, lse: torch.Tensor, q_seq_idx: Optional[torch.Tensor] = None,
                              seq_lens: Optional[torch.Tensor] = None, err_word: Optional[torch.Tensor] = None,
                              stream=None):
    """sparse_mla_decode for callers that cannot allocate: out (bf16
    [T,H,512]) and lse (fp32 [T,H]) are required, the split partials go to the
    library's own scratch, and neither this function nor the library
    allocates GPU memory. Calls that overlap on the GPU share that scratch
    and race. Returns (out, lse)."""
    _need(q_latent, "q_latent", torch.bfloat16, 3)
    _need(q_rope, "q_rope", torch.bfloat16, 3)
    _need(cache, "cache", torch.uint8, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    T, H, dl = q_latent.shape
    if dl != 512 or tuple(q_rope.shape) != (T, H, 64):
        raise ValueError("q_latent must be [T, H, 512] and q_rope [T, H, 64]")
    if topk_idx.shape[0] != T or tuple(out.shape) != (T, H, 512) or tuple(lse.shape) != (T, H):
        raise ValueError("topk_idx must be [T, topk], out [T, H, 512] and lse [T, H]")
    if cache.shape[1:] != (PAGE_TOKENS, ROW_BYTES):
        raise ValueError("cache must be [num_pages, 64, 352]")
    if q_seq_idx is not None:
        _need(q_seq_idx, "q_seq_idx", torch.int32, 1)
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, 1)
    lib = load()
    _check(lib.sparse_mla_decode_noalloc(_ptr(q_latent), _ptr(q_rope), _ptr(cache), cache.shape[0],
                                         _ptr(block_table), block_table.shape[0], block_table.shape[1],
                                         _ptr(topk_idx), topk_idx.shape[1], _ptr(q_seq_idx), _ptr(seq_lens), T, H,
                                         float(sm_scale), _ptr(out), _ptr(lse), _ptr(err_word),
                                         _stream(q_latent, stream)))
    return out, lse


def nvfp4_stage_dequant_fp8(cache: torch.Tensor, block_table: torch.Tensor, topk_idx: torch.Tensor,
                            q_seq_idx: Optional[torch.Tensor] = None, seq_lens: Optional[torch.Tensor] = None,
                            fp8_rows: Optional[torch.Tensor] = None, row_idx: Optional[torch.Tensor] = None,
                            err_word: Optional[torch.Tensor] = None, stream=None):
    """Staged baseline, stage 1: -> (fp8_rows uint8 [T,topk,576], row_idx
    int32 [T,topk])."""
    _need(cache, "cache", torch.uint8, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    T, topk = topk_idx.shape
    if fp8_rows is None:
        fp8_rows = torch.empty((T, topk, FP8_ROW_BYTES), dtype=torch.uint8, device=cache.device)
    if row_idx is None:
        row_idx = torch.empty((T, topk), dtype=torch.int32, device=cache.device)
    _need(fp8_rows, "fp8_rows", torch.uint8, 3)
    _need(row_idx, "row_idx", torch.int32, 2)
    lib = load()
    _check(lib.nvfp4_stage_dequant_fp8(_ptr(cache), cache.shape[0], _ptr(block_table), block_table.shape[0],
                                       block_table.shape[1], _ptr(topk_idx), topk, _ptr(q_seq_idx), _ptr(seq_lens),
                                       T, _ptr(fp8_rows), _ptr(row_idx), _ptr(err_word), _stream(cache, stream)))
    return fp8_rows, row_idx


def sparse_mla_decode_fp8rows(q_latent: torch.Tensor, q_rope: torch.Tensor, fp8_rows: torch.Tensor,
                              row_idx: torch.Tensor, sm_scale: float, out: Optional[torch.Tensor] = None,
                              lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                              err_word: Optional[torch.Tensor] = None, impl=None, num_splits=None, stream=None):
    """Staged baseline, stage 2 (attention over 576-byte FP8 rows)."""
    _need(q_latent, "q_latent", torch.bfloat16, 3)
    _need(q_rope, "q_rope", torch.bfloat16, 3)
    _need(fp8_rows, "fp8_rows", torch.uint8, 3)
    _need(row_idx, "row_idx", torch.int32, 2)
    T, H, _ = q_latent.shape
    topk = row_idx.shape[1]
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q_latent.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q_latent.device)
    opts = _opts(impl, num_splits)
    lib = load()
    if workspace is None:
        nbytes = int(lib.sparse_mla_decode_fp8rows_workspace_size(T, H, topk, opts))
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q_latent.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sparse_mla_decode_fp8rows(_ptr(q_latent), _ptr(q_rope), _ptr(fp8_rows), _ptr(row_idx), topk, T, H,
                                         float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                         _ptr(err_word), opts, _stream(q_latent, stream)))
    return out, lse


# short names of the two calls of the path (the same functions)
pack = nvfp4_mla_pack
decode = sparse_mla_decode
