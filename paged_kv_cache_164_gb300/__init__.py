"""pkv — decode-phase attention over a paged KV cache on NVIDIA GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/pkv.h`` (``libpkv.so``).
Every step of the path runs in the library's CUDA kernels; this module only
checks tensor types, passes device pointers, sizes and the current CUDA stream,
and turns status codes into exceptions.  PyTorch provides device memory and
streams.  There is no CPU fallback: if the library is not built, or a tensor is
not on a CUDA device, the call raises.

Calls (same names as the C entry points, without the ``pkv_`` prefix):

  append(k_new, v_new, k_cache, v_cache, slot_mapping)
  decode_attention(q, k_cache, v_cache, block_tables, context_lens, max_context_len)
  merge(partial_o, partial_lse)
  gather(k_cache, v_cache, block_tables, context_lens, max_context_len)
  check_error(err_flag)
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# The in-tree build; PKV_LIBRARY may point at another build of the same library.
LIB_PATH = os.environ.get("PKV_LIBRARY") or os.path.join(_HERE, "_build", "libpkv.so")

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                3: "PKV_ERR_WORKSPACE", 4: "PKV_ERR_CUDA", 5: "PKV_ERR_DEVICE_INDEX",
                6: "PKV_ERR_DEVICE_TIMEOUT"}
EFLAG_BLOCK_ID, EFLAG_SLOT, EFLAG_CONTEXT_LEN, EFLAG_TIMEOUT, EFLAG_GROUP = 0x1, 0x2, 0x4, 0x8, 0x10
MAX_SPLITS = 1024
_DTYPES = {torch.float16: 0, torch.bfloat16: 1}
SIZE_MAX = ctypes.c_size_t(-1).value


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads ``libpkv.so`` (once) and declares the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"pkv CUDA library not built: {path} is missing "
                          "(run `python -m paged_kv_cache_164_gb300.build`)")
    lib = ctypes.CDLL(path)
    p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.pkv_append.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, p]
    lib.pkv_decode_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.pkv_decode_workspace_size.restype = sz
    lib.pkv_decode_num_splits.argtypes = [i, i, i, i, i, i, i]
    lib.pkv_decode_num_splits.restype = i
    lib.pkv_decode_num_splits_fp8.argtypes = [i, i, i, i, i, i, i]
    lib.pkv_decode_num_splits_fp8.restype = i
    lib.pkv_decode_attention.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, f, i, p, sz,
                                         i, p, p]
    lib.pkv_append_decode_attention.argtypes = [p, p, p, p, p, p, p, i, p, i, i, i, i, i, i, i,
                                                f, i, p, sz, i, p, p]
    lib.pkv_append_decode_attention_fp8.argtypes = [p, p, p, p, p, p, p, i, p, i, i, i, i, i, i,
                                                    i, f, f, f, i, p, sz, i, p, p]
    lib.pkv_append_fp8.argtypes = [p, p, p, p, p, i, i, i, i, i, f, f, i, p, p]
    lib.pkv_decode_attention_fp8.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, f, f, f, i,
                                             p, sz, i, p, p]
    lib.pkv_decode_attention_noalloc.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, f,
                                                 i, i, p, p]
    lib.pkv_prefix_shared_workspace_size.argtypes = [i, i, i, i, i, i, i, i, i]
    lib.pkv_prefix_shared_workspace_size.restype = sz
    lib.pkv_decode_attention_prefix_shared.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, f,
                                                       i, p, p, i, i, p, sz, i, p, p]
    lib.pkv_multi_query_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.pkv_multi_query_workspace_size.restype = sz
    lib.pkv_multi_query_plan.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
    lib.pkv_multi_query_attention.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, i, f, p,
                                              sz, i, p, p]
    lib.pkv_merge.argtypes = [p, p, p, i, i, i, i, i, p]
    lib.pkv_gather.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i, i, p, p]
    lib.pkv_check_error.argtypes = [p, p, ctypes.POINTER(ctypes.c_int32)]
    lib.pkv_status_string.argtypes = [i]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_max_group_size.argtypes = []
    lib.pkv_debug_build.argtypes = []
    lib.pkv_debug_build.restype = i
    lib.pkv_selftest_wait_timeout.argtypes = [p, ctypes.c_ulonglong, p]
    for name in ("pkv_append", "pkv_decode_attention", "pkv_decode_attention_noalloc",
                 "pkv_append_decode_attention", "pkv_append_decode_attention_fp8",
                 "pkv_append_fp8", "pkv_decode_attention_fp8",
                 "pkv_decode_attention_prefix_shared", "pkv_multi_query_attention",
                 "pkv_merge", "pkv_gather", "pkv_selftest_wait_timeout",
                 "pkv_check_error", "pkv_max_group_size", "pkv_multi_query_plan"):
        getattr(lib, name).restype = i
    _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, what)


def _dev(t: torch.Tensor, name: str, dtype=None) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _opt(t: Optional[torch.Tensor], name: str) -> ctypes.c_void_p:
    return ctypes.c_void_p(0) if t is None else _dev(t, name, torch.int32)


def _stream(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _kv_dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"KV dtype must be float16 or bfloat16, got {t.dtype}")
    return _DTYPES[t.dtype]


LAYOUT_HND = 0x100
_LAYOUTS = ("nhd", "hnd")


def _cache_dims(k_cache: torch.Tensor, layout: str):
    """(num_blocks, block_size, num_kv_heads, head_dim) of a token-major ("nhd",
    [blocks][bs][H_kv][d]) or head-major ("hnd", [blocks][H_kv][bs][d]) cache."""
    if layout not in _LAYOUTS:
        raise ValueError(f"layout must be one of {_LAYOUTS}, got {layout!r}")
    if k_cache.dim() != 4:
        raise ValueError("a cache is 4-D")
    nb, a, c, d = k_cache.shape
    return (nb, a, c, d) if layout == "nhd" else (nb, c, a, d)


def _kv_code(k_cache: torch.Tensor, layout: str) -> int:
    """The dtype argument for a call that takes the cache: element type plus layout flag."""
    return _kv_dtype(k_cache) | (LAYOUT_HND if layout == "hnd" else 0)


def new_error_flag(device) -> torch.Tensor:
    """A zeroed int32 device word for the kernels' index/timeout flags."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
           v_cache: torch.Tensor, slot_mapping: torch.Tensor,
           err_flag: Optional[torch.Tensor] = None, stream=None, layout: str = "nhd") -> None:
    """Scatters k_new/v_new [T, H_kv, d] into the caches at ``slot_mapping`` (int64 [T])."""
    lib = load()
    nb, bs, h_kv, d = _cache_dims(k_cache, layout)
    if v_cache.shape != k_cache.shape or k_new.shape[1:] != (h_kv, d) or \
            v_new.shape != k_new.shape or slot_mapping.shape != (k_new.shape[0],):
        raise ValueError("inconsistent append shapes")
    dt = k_cache.dtype
    st = lib.pkv_append(_dev(k_new, "k_new", dt), _dev(v_new, "v_new", dt),
                        _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt),
                        _dev(slot_mapping, "slot_mapping", torch.int64), k_new.shape[0], nb, bs,
                        h_kv, d, _kv_code(k_cache, layout), _opt(err_flag, "err_flag"),
                        _stream(stream, k_cache.device))
    _check(st, "pkv_append")


def workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                   block_size: int, max_context_len: int, num_splits: int = 0) -> int:
    """Bytes of workspace ``decode_attention`` needs (0 if none) on the current device."""
    n = load().pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                         block_size, max_context_len, num_splits)
    if n == SIZE_MAX:
        raise PkvError(1, "pkv_decode_workspace_size")
    return int(n)


def decode_num_splits(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                      block_size: int, max_context_len: int, num_splits: int = 0,
                      kv: str = "16bit") -> int:
    """KV partitions per sequence ``decode_attention`` (kv="16bit") or
    ``decode_attention_fp8`` (kv="fp8") uses on the current device."""
    lib = load()
    fn = lib.pkv_decode_num_splits_fp8 if kv == "fp8" else lib.pkv_decode_num_splits
    n = fn(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len, num_splits)
    if n < 0:
        raise PkvError(1, "pkv_decode_num_splits")
    return int(n)


def decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     block_tables: torch.Tensor, context_lens: torch.Tensor,
                     max_context_len: int, scale: Optional[float] = None, num_splits: int = 0,
                     out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     err_flag: Optional[torch.Tensor] = None, stream=None,
                     layout: str = "nhd") -> torch.Tensor:
    """softmax(q K^T * scale) V per sequence and query head over the paged cache.

    q [B, H_q, d]; caches [num_blocks, bs, H_kv, d]; block_tables int32
    [B, max_blocks]; context_lens int32 [B] (device); scale defaults to
    1/sqrt(d).  ``workspace`` (uint8, device) is allocated when not given.
    """
    lib = load()
    b, h_q, d = q.shape
    nb, bs, h_kv, d2 = _cache_dims(k_cache, layout)
    if d2 != d or v_cache.shape != k_cache.shape or block_tables.dim() != 2 or \
            block_tables.shape[0] != b or context_lens.shape != (b,):
        raise ValueError("inconsistent decode shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dt = k_cache.dtype
    if out is None:
        out = torch.empty_like(q)
    # a given workspace is checked against the plan by the library itself
    need = workspace_size(b, h_q, h_kv, d, bs, max_context_len, num_splits) \
        if workspace is None else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(0) if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.pkv_decode_attention(
        _dev(out, "out", dt), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32),
        int(max_context_len), b, nb, bs, h_q, h_kv, d, float(scale), int(num_splits), ws_ptr,
        ws_bytes, _kv_code(k_cache, layout), _opt(err_flag, "err_flag"), _stream(stream, q.device))
    _check(st, "pkv_decode_attention")
    return out


def append_decode_attention(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                            k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor,
                            max_context_len: int, scale: Optional[float] = None,
                            num_splits: int = 0, out: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None,
                            err_flag: Optional[torch.Tensor] = None, stream=None,
                            layout: str = "nhd") -> torch.Tensor:
    """One decode step in one launch: sequence b's new token (k_new[b], v_new[b],
    [B, H_kv, d]) is written at position context_lens[b] - 1 of its block table,
    then ``decode_attention`` runs over the updated cache."""
    lib = load()
    b, h_q, d = q.shape
    nb, bs, h_kv, d2 = _cache_dims(k_cache, layout)
    if d2 != d or v_cache.shape != k_cache.shape or block_tables.dim() != 2 or \
            block_tables.shape[0] != b or context_lens.shape != (b,) or \
            k_new.shape != (b, h_kv, d) or v_new.shape != (b, h_kv, d):
        raise ValueError("inconsistent append-decode shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dt = k_cache.dtype
    if out is None:
        out = torch.empty_like(q)
    # a given workspace is checked against the plan by the library itself
    need = workspace_size(b, h_q, h_kv, d, bs, max_context_len, num_splits) \
        if workspace is None else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(0) if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.pkv_append_decode_attention(
        _dev(out, "out", dt), _dev(q, "q", dt), _dev(k_new, "k_new", dt), _dev(v_new, "v_new", dt),
        _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), b, nb, bs, h_q,
        h_kv, d, float(scale), int(num_splits), ws_ptr, ws_bytes, _kv_code(k_cache, layout),
        _opt(err_flag, "err_flag"), _stream(stream, q.device))
    _check(st, "pkv_append_decode_attention")
    return out


def append_fp8(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
               v_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float, v_scale: float,
               err_flag: Optional[torch.Tensor] = None, stream=None,
               layout: str = "nhd") -> None:
    """Quantising append into uint8 E4M3 caches: element x of a new K row is
    stored as E4M3(x / k_scale) (nearest, ties to even, saturating at +-448)."""
    lib = load()
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("E4M3 caches are uint8 tensors of codes")
    nb, bs, h_kv, d = _cache_dims(k_cache, layout)
    if v_cache.shape != k_cache.shape or k_new.shape[1:] != (h_kv, d) or \
            v_new.shape != k_new.shape or slot_mapping.shape != (k_new.shape[0],):
        raise ValueError("inconsistent fp8 append shapes")
    st = lib.pkv_append_fp8(_dev(k_new, "k_new"), _dev(v_new, "v_new"),
                            _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                            _dev(slot_mapping, "slot_mapping", torch.int64), k_new.shape[0], nb,
                            bs, h_kv, d, float(k_scale), float(v_scale),
                            _kv_code(k_new, layout), _opt(err_flag, "err_flag"),
                            _stream(stream, k_cache.device))
    _check(st, "pkv_append_fp8")


def decode_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_tables: torch.Tensor, context_lens: torch.Tensor,
                         max_context_len: int, k_scale: float, v_scale: float,
                         scale: Optional[float] = None, num_splits: int = 0,
                         out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         err_flag: Optional[torch.Tensor] = None, stream=None,
                         layout: str = "nhd") -> torch.Tensor:
    """``decode_attention`` over uint8 E4M3 caches whose codes stand for
    code * k_scale and code * v_scale; q (and out) fp16 or bf16; head_dim 128."""
    lib = load()
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("E4M3 caches are uint8 tensors of codes")
    b, h_q, d = q.shape
    nb, bs, h_kv, d2 = _cache_dims(k_cache, layout)
    if d2 != d or v_cache.shape != k_cache.shape or block_tables.dim() != 2 or \
            block_tables.shape[0] != b or context_lens.shape != (b,):
        raise ValueError("inconsistent fp8 decode shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    # a given workspace is checked against the plan by the library itself
    need = workspace_size(b, h_q, h_kv, d, bs, max_context_len, num_splits) \
        if workspace is None else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(0) if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.pkv_decode_attention_fp8(
        _dev(out, "out", q.dtype), _dev(q, "q"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32),
        int(max_context_len), b, nb, bs, h_q, h_kv, d, float(scale), float(k_scale),
        float(v_scale), int(num_splits), ws_ptr, ws_bytes, _kv_code(q, layout),
        _opt(err_flag, "err_flag"), _stream(stream, q.device))
    _check(st, "pkv_decode_attention_fp8")
    return out


def append_decode_attention_fp8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor,
                                max_context_len: int, k_scale: float, v_scale: float,
                                scale: Optional[float] = None, num_splits: int = 0,
                                out: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None,
                                err_flag: Optional[torch.Tensor] = None, stream=None,
                                layout: str = "nhd") -> torch.Tensor:
    """``append_decode_attention`` over uint8 E4M3 caches: sequence b's new token
    is quantised as ``append_fp8`` does and written at position context_lens[b] - 1,
    then ``decode_attention_fp8`` runs over the updated cache; head_dim 128."""
    lib = load()
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("E4M3 caches are uint8 tensors of codes")
    b, h_q, d = q.shape
    nb, bs, h_kv, d2 = _cache_dims(k_cache, layout)
    if d2 != d or v_cache.shape != k_cache.shape or block_tables.dim() != 2 or \
            block_tables.shape[0] != b or context_lens.shape != (b,) or \
            k_new.shape != (b, h_kv, d) or v_new.shape != (b, h_kv, d):
        raise ValueError("inconsistent fp8 append-decode shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    # a given workspace is checked against the plan by the library itself
    need = workspace_size(b, h_q, h_kv, d, bs, max_context_len, num_splits) \
        if workspace is None else 0
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = ctypes.c_void_p(0) if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.pkv_append_decode_attention_fp8(
        _dev(out, "out", q.dtype), _dev(q, "q"), _dev(k_new, "k_new", q.dtype),
        _dev(v_new, "v_new", q.dtype), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), b, nb, bs, h_q,
        h_kv, d, float(scale), float(k_scale), float(v_scale), int(num_splits), ws_ptr,
        ws_bytes, _kv_code(q, layout), _opt(err_flag, "err_flag"), _stream(stream, q.device))
    _check(st, "pkv_append_decode_attention_fp8")
    return out


def prefix_shared_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                 head_dim: int, block_size: int, max_context_len: int,
                                 num_groups: int, max_group_size: int, max_prefix_len: int) -> int:
    """Bytes of workspace ``decode_attention_prefix_shared`` needs on the current device."""
    n = load().pkv_prefix_shared_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                block_size, max_context_len, num_groups,
                                                max_group_size, max_prefix_len)
    if n == SIZE_MAX:
        raise PkvError(1, "pkv_prefix_shared_workspace_size")
    return int(n)


def decode_attention_prefix_shared(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                   block_tables: torch.Tensor, context_lens: torch.Tensor,
                                   max_context_len: int, group_start: torch.Tensor,
                                   group_prefix_len: torch.Tensor, max_group_size: int,
                                   max_prefix_len: int, scale: Optional[float] = None,
                                   out: Optional[torch.Tensor] = None,
                                   workspace: Optional[torch.Tensor] = None,
                                   err_flag: Optional[torch.Tensor] = None,
                                   stream=None, layout: str = "nhd") -> torch.Tensor:
    """``decode_attention`` for batches whose sequences share prompt-prefix blocks.

    group_start int32 [G+1] and group_prefix_len int32 [G] (device) describe
    contiguous groups of sequences whose first group_prefix_len[p] tokens are
    the same physical blocks; each group's prefix is read once for all members.
    Inside the call the prefix kernel runs on a second stream of the library's
    own, forked from ``stream`` and joined back to it before the call returns,
    so work queued on ``stream`` before and after is ordered as usual.
    """
    lib = load()
    b, h_q, d = q.shape
    nb, bs, h_kv, d2 = _cache_dims(k_cache, layout)
    ng = group_prefix_len.shape[0]
    if d2 != d or v_cache.shape != k_cache.shape or block_tables.dim() != 2 or \
            block_tables.shape[0] != b or context_lens.shape != (b,) or \
            group_start.shape != (ng + 1,):
        raise ValueError("inconsistent shared-prefix decode shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dt = k_cache.dtype
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:  # a given workspace is checked by the library itself
        need = prefix_shared_workspace_size(b, h_q, h_kv, d, bs, max_context_len, ng,
                                            max_group_size, max_prefix_len)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = lib.pkv_decode_attention_prefix_shared(
        _dev(out, "out", dt), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32),
        int(max_context_len), b, nb, bs, h_q, h_kv, d, float(scale), ng,
        _dev(group_start, "group_start", torch.int32),
        _dev(group_prefix_len, "group_prefix_len", torch.int32), int(max_group_size),
        int(max_prefix_len), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _kv_code(k_cache, layout),
        _opt(err_flag, "err_flag"), _stream(stream, q.device))
    _check(st, "pkv_decode_attention_prefix_shared")
    return out


def multi_query_plan(num_seqs: int, q_len: int, num_q_heads: int, num_kv_heads: int,
                     head_dim: int, block_size: int, max_context_len: int) -> tuple:
    """(kernel, context partitions) of a ``multi_query_attention`` call on the
    current device: kernel "decode" (at most twice ``pkv_max_group_size()``, 32,
    query rows per sequence and KV head) or "tcgen05"."""
    parts = ctypes.c_int(0)
    r = load().pkv_multi_query_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
                                    block_size, max_context_len, ctypes.byref(parts))
    if r < 0:
        raise PkvError(1, "pkv_multi_query_plan")
    return ("decode" if r == 1 else "tcgen05"), int(parts.value)


def multi_query_workspace_size(num_seqs: int, q_len: int, num_q_heads: int, num_kv_heads: int,
                               head_dim: int, block_size: int, max_context_len: int) -> int:
    """Bytes of workspace ``multi_query_attention`` needs on the current device."""
    n = load().pkv_multi_query_workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads,
                                              head_dim, block_size, max_context_len)
    if n == SIZE_MAX:
        raise PkvError(1, "pkv_multi_query_workspace_size")
    return int(n)


def multi_query_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_tables: torch.Tensor, context_lens: torch.Tensor,
                          max_context_len: int, scale: Optional[float] = None,
                          out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None,
                          err_flag: Optional[torch.Tensor] = None, stream=None,
                          layout: str = "nhd") -> torch.Tensor:
    """Causal attention of q_len new query tokens per sequence over the paged cache.

    q [B, q_len, H_q, d]; context_lens counts the cached tokens including the
    q_len new ones (appended first); query token i of sequence b attends to
    positions 0 .. context_lens[b] - q_len + i.
    """
    lib = load()
    b, q_len, h_q, d = q.shape
    nb, bs, h_kv, d2 = _cache_dims(k_cache, layout)
    if d2 != d or v_cache.shape != k_cache.shape or block_tables.dim() != 2 or \
            block_tables.shape[0] != b or context_lens.shape != (b,):
        raise ValueError("inconsistent multi-query shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dt = k_cache.dtype
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:  # a given workspace is checked by the library itself
        need = multi_query_workspace_size(b, q_len, h_q, h_kv, d, bs, max_context_len)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = lib.pkv_multi_query_attention(
        _dev(out, "out", dt), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32),
        int(max_context_len), b, q_len, nb, bs, h_q, h_kv, d, float(scale),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _kv_code(k_cache, layout), _opt(err_flag, "err_flag"), _stream(stream, q.device))
    _check(st, "pkv_multi_query_attention")
    return out


NOALLOC_SCRATCH_BYTES = 8 << 20


def decode_attention_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             block_tables: torch.Tensor, context_lens: torch.Tensor,
                             max_context_len: int, out: torch.Tensor,
                             scale: Optional[float] = None, num_splits: int = 0,
                             err_flag: Optional[torch.Tensor] = None, stream=None,
                             layout: str = "nhd") -> torch.Tensor:
    """``decode_attention`` for callers that cannot allocate device memory.

    Same result, but the split-K scratch is a fixed 8 MiB array inside the
    library (reserved per GPU for the life of the process) and the caller
    passes ``out``, so the call allocates nothing.  Calls share that array:
    keep calls that use it ordered on one stream.  The first call in each CUDA
    context (normally once per device) looks the array's address up; make it
    before any stream capture.  Plans needing more scratch than the array
    holds are rejected (PKV_ERR_WORKSPACE); ask for fewer splits then.
    """
    lib = load()
    b, h_q, d = q.shape
    nb, bs, h_kv, d2 = _cache_dims(k_cache, layout)
    if d2 != d or v_cache.shape != k_cache.shape or block_tables.dim() != 2 or \
            block_tables.shape[0] != b or context_lens.shape != (b,) or out.shape != q.shape:
        raise ValueError("inconsistent decode shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dt = k_cache.dtype
    st = lib.pkv_decode_attention_noalloc(
        _dev(out, "out", dt), _dev(q, "q", dt), _dev(k_cache, "k_cache", dt),
        _dev(v_cache, "v_cache", dt), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32),
        int(max_context_len), b, nb, bs, h_q, h_kv, d, float(scale), int(num_splits),
        _kv_code(k_cache, layout), _opt(err_flag, "err_flag"), _stream(stream, q.device))
    _check(st, "pkv_decode_attention_noalloc")
    return out


def merge(partial_o: torch.Tensor, partial_lse: torch.Tensor, out_dtype=torch.bfloat16,
          out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Log-sum-exp merge: partial_o fp32 [B, H_q, P, d], partial_lse fp32 [B, H_q, P]."""
    lib = load()
    b, h_q, p_, d = partial_o.shape
    if partial_lse.shape != (b, h_q, p_):
        raise ValueError("inconsistent merge shapes")
    if out is None:
        out = torch.empty((b, h_q, d), dtype=out_dtype, device=partial_o.device)
    st = lib.pkv_merge(_dev(out, "out", out.dtype),
                       _dev(partial_o, "partial_o", torch.float32),
                       _dev(partial_lse, "partial_lse", torch.float32), b, h_q, p_, d,
                       _kv_dtype(out), _stream(stream, partial_o.device))
    _check(st, "pkv_merge")
    return out


def gather(k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
           context_lens: torch.Tensor, max_context_len: int,
           k_out: Optional[torch.Tensor] = None, v_out: Optional[torch.Tensor] = None,
           err_flag: Optional[torch.Tensor] = None, stream=None, layout: str = "nhd"):
    """Contiguous copies [B, max_context_len, H_kv, d] of each sequence's cached K and V."""
    lib = load()
    nb, bs, h_kv, d = _cache_dims(k_cache, layout)
    b = block_tables.shape[0]
    shape = (b, max_context_len, h_kv, d)
    if k_out is None:
        k_out = torch.zeros(shape, dtype=k_cache.dtype, device=k_cache.device)
    if v_out is None:
        v_out = torch.zeros(shape, dtype=k_cache.dtype, device=k_cache.device)
    dt = k_cache.dtype
    st = lib.pkv_gather(_dev(k_out, "k_out", dt), _dev(v_out, "v_out", dt),
                        _dev(k_cache, "k_cache", dt), _dev(v_cache, "v_cache", dt),
                        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                        _dev(context_lens, "context_lens", torch.int32), int(max_context_len),
                        b, nb, bs, h_kv, d, _kv_code(k_cache, layout), _opt(err_flag, "err_flag"),
                        _stream(stream, k_cache.device))
    _check(st, "pkv_gather")
    return k_out, v_out


def check_error(err_flag: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the device error word (0 = no error)."""
    lib = load()
    word = ctypes.c_int32(0)
    st = lib.pkv_check_error(_dev(err_flag, "err_flag", torch.int32),
                             _stream(stream, err_flag.device), ctypes.byref(word))
    if st not in (0, 5, 6):
        raise PkvError(st, "pkv_check_error")
    return int(word.value)


def selftest_wait_timeout(err_flag: torch.Tensor, limit_ns: int = 20_000_000, stream=None) -> None:
    """Runs the bounded-wait self-test kernel (see pkv.h); the flag then reads EFLAG_TIMEOUT."""
    st = load().pkv_selftest_wait_timeout(_dev(err_flag, "err_flag", torch.int32), int(limit_ns),
                                          _stream(stream, err_flag.device))
    _check(st, "pkv_selftest_wait_timeout")


def status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()
