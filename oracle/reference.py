"""Oracle functions — TEST INFRASTRUCTURE ONLY (see the package docstring).

Two implementations of decode attention over a paged cache live here:

* ``decode_attention`` — the C oracle (``pkv_oracle.c``, fp64, OpenMP over
  (sequence, query head)); fast enough for the full benchmark shapes;
* ``decode_attention_np`` — the same definition written out with numpy, per
  (sequence, query head), for small cases;

plus the pages' own per-page formulation (``segment_partials`` and
``combine_result``), the log-sum-exp merge of split partials (``merge_lse``),
the host scatter (``append``), the host gather (``gather_kv``) and the KV-size
closed form (``kv_cache_bytes``).

All arrays are numpy.  16-bit cache contents are passed as their raw ``uint16``
bit patterns together with a dtype name ("fp16" or "bf16"); the oracle decodes
them itself.
"""
from __future__ import annotations

import ctypes
import math
from typing import Sequence

import numpy as np

from . import build as _build

DTYPE_CODES = {"fp16": 0, "bf16": 1}

_LIB = None


def load_library(path: str) -> ctypes.CDLL:
    """Loads a compiled oracle shared object and declares its C signatures."""
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_decode_values.argtypes = [p, p, ctypes.c_int64, i]
    lib.oracle_decode_values.restype = None
    lib.oracle_decode_attention.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i,
                                            ctypes.c_double, i]
    lib.oracle_decode_attention.restype = i
    lib.oracle_append.argtypes = [p, p, p, p, p, i, i, i, i, i]
    lib.oracle_append.restype = i
    lib.oracle_decode_e4m3.argtypes = [p, p, ctypes.c_int64]
    lib.oracle_decode_e4m3.restype = None
    lib.oracle_encode_e4m3.argtypes = [p, p, ctypes.c_int64]
    lib.oracle_encode_e4m3.restype = None
    lib.oracle_append_fp8.argtypes = [p, p, p, p, p, i, i, i, i, i, ctypes.c_float,
                                      ctypes.c_float, i]
    lib.oracle_append_fp8.restype = i
    lib.oracle_decode_attention_fp8.argtypes = [p, p, p, p, p, i, p, i, i, i, i, i, i,
                                                ctypes.c_double, ctypes.c_double,
                                                ctypes.c_double, i]
    lib.oracle_decode_attention_fp8.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    return lib


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load_library(_build.build())
    return _LIB


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected raw uint16 bit patterns, got {a.dtype}")
    return a


def num_threads() -> int:
    """Threads the C oracle's OpenMP loops use."""
    return int(_lib().oracle_num_threads())


def decode_values(bits: np.ndarray, dtype: str, lib: ctypes.CDLL = None) -> np.ndarray:
    """Exact float64 values of fp16 / bf16 bit patterns (the oracle's own decoder)."""
    bits = _bits(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    (lib or _lib()).oracle_decode_values(_ptr(out), _ptr(bits), bits.size, DTYPE_CODES[dtype])
    return out


# ---------------------------------------------------------------------------
# Closed form for the cache size
# ---------------------------------------------------------------------------

def kv_cache_bytes(num_layers: int, num_kv_heads: int, head_dim: int, seq_len: int,
                   batch: int, dtype_size: int) -> int:
    """KV-cache bytes = 2 * L * H * d_h * S * B * dtype_size.

    The factor 2 counts K and V; H is the number of KV heads (inference.html,
    "KV Cache 的显存计算").  With H * d_h = hidden size and S = B = 1 this is the
    per-token form 2 * layers * hidden * bytes (gsyq.cn essay, §三).
    """
    return 2 * num_layers * num_kv_heads * head_dim * seq_len * batch * dtype_size


# ---------------------------------------------------------------------------
# Append and gather
# ---------------------------------------------------------------------------

def append(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
           slot_mapping: np.ndarray, lib: ctypes.CDLL = None) -> int:
    """Host scatter, in place: token i goes to block slot//bs, offset slot%bs; slot < 0 skips.

    Caches are uint16 [num_blocks, block_size, num_kv_heads, head_dim]; k_new and
    v_new are uint16 [num_tokens, num_kv_heads, head_dim]; slot_mapping is int64.
    Returns 0, or -2 if some slot lies beyond the pool (that token is skipped).
    (inference.html, KVCachePool.write_tokens; tutorial chapter 12,
    PagedKVCache.update.)  ``lib`` selects another build of the C oracle.
    """
    for a in (k_cache, v_cache):
        if a.dtype != np.uint16 or not a.flags.c_contiguous:
            raise TypeError("caches must be contiguous uint16 arrays (updated in place)")
    num_blocks, block_size, h_kv, d = k_cache.shape
    k_new = _bits(k_new)
    v_new = _bits(v_new)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return int((lib or _lib()).oracle_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                    _ptr(slots), int(slots.size), num_blocks, block_size,
                                    h_kv, d))


def gather_kv(k_cache: np.ndarray, v_cache: np.ndarray, block_tables: np.ndarray,
              context_len: int, seq: int, kv_head: int) -> tuple[np.ndarray, np.ndarray]:
    """Contiguous [n, d] copies of one sequence's K and V rows for one KV head.

    Token t is read from block block_tables[seq, t // bs] at offset t % bs
    (gsyq.cn essay, §三.2 get_kv_cache; tutorial chapter 12, PagedKVCache.update).
    Works on any element type; the copy is exact.
    """
    bs = k_cache.shape[1]
    t = np.arange(context_len)
    blk = block_tables[seq, t // bs].astype(np.int64)
    off = t % bs
    return k_cache[blk, off, kv_head, :].copy(), v_cache[blk, off, kv_head, :].copy()


# ---------------------------------------------------------------------------
# Decode attention: the plain definition
# ---------------------------------------------------------------------------

def decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                     dtype: str, lib: ctypes.CDLL = None) -> np.ndarray:
    """C oracle: out[b, h] = softmax(scale * q[b, h] . K_t) weighted sum of V_t, fp64.

    q: uint16 [B, H_q, d]; caches uint16 [num_blocks, bs, H_kv, d];
    block_tables int32 [B, max_blocks]; context_lens int32 [B].  Returns float64
    [B, H_q, d].  Query head h reads KV head h // (H_q / H_kv).
    Raises ValueError when a block id that would be read is out of range.
    ``lib`` selects another build of the C oracle (the tests use it to check
    that deliberately broken copies fail the pins).
    """
    q = _bits(q)
    k_cache = _bits(k_cache)
    v_cache = _bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, h_q, d = q.shape
    num_blocks, bs, h_kv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape or cl.shape != (num_seqs,):
        raise ValueError("inconsistent shapes")
    out = np.empty((num_seqs, h_q, d), dtype=np.float64)
    rc = (lib or _lib()).oracle_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), int(bt.shape[1]), _ptr(cl),
        num_seqs, num_blocks, bs, h_q, h_kv, d, float(scale), DTYPE_CODES[dtype])
    if rc == -1:
        raise ValueError("invalid arguments")
    if rc == -2:
        raise ValueError("block id out of range")
    return out


def multi_query_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                          block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                          dtype: str, lib: ctypes.CDLL = None) -> np.ndarray:
    """Causal attention of q_len new query tokens per sequence, fp64.

    q: uint16 [B, q_len, H_q, d]; the chunk's K/V are already in the cache and
    counted by context_lens.  Query token i of sequence b attends to positions
    0 .. n_b - q_len + i: a chunked-prefill chunk's queries see the cached KV
    and the chunk's own KV up to their own position (LLM-101-CN "推理优化",
    Chunked Prefill; each query attends to keys up to its own position, tutorial
    chapter 12, Attention(Q_t, K_1:t, V_1:t)).  That is the decode-attention
    definition applied to every query token with its own causal context length
    (at least 0).  Returns float64 [B, q_len, H_q, d].
    """
    q = _bits(q)
    num_seqs, q_len, h_q, d = q.shape
    cl = np.asarray(context_lens, dtype=np.int64)
    if cl.shape != (num_seqs,):
        raise ValueError("inconsistent shapes")
    limits = cl[:, None] - q_len + 1 + np.arange(q_len)[None, :]
    rows = decode_attention(q.reshape(num_seqs * q_len, h_q, d), k_cache, v_cache,
                            np.repeat(np.asarray(block_tables), q_len, axis=0),
                            np.maximum(limits, 0).reshape(-1).astype(np.int32), scale, dtype,
                            lib=lib)
    return rows.reshape(num_seqs, q_len, h_q, d)


def decode_e4m3(codes: np.ndarray, lib: ctypes.CDLL = None) -> np.ndarray:
    """Exact float64 values of E4M3 codes (1 sign, 4 exponent bits with bias 7,
    3 fraction bits, no infinities, S.1111.111 = NaN): the oracle's own decoder."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    (lib or _lib()).oracle_decode_e4m3(_ptr(out), _ptr(c), int(c.size))
    return out


def encode_e4m3(x: np.ndarray, lib: ctypes.CDLL = None) -> np.ndarray:
    """E4M3 codes of float32 values: round to nearest, ties to even, saturating
    at +-448 (NaN gives 0x7F)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint8)
    (lib or _lib()).oracle_encode_e4m3(_ptr(out), _ptr(f), int(f.size))
    return out


def append_fp8(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
               slot_mapping: np.ndarray, k_scale: float, v_scale: float, dtype: str,
               lib: ctypes.CDLL = None) -> int:
    """Quantising host scatter, in place, into uint8 E4M3 caches
    [num_blocks, bs, H_kv, d]: element x of the new K row is stored as
    E4M3(x / k_scale), the quotient in fp32 (vLLM deep dive, 3.3 FP8 inference:
    E4M3 with the range held by a scale; 2.2: KV-cache write fused with
    quantisation).  Returns 0, or -2 if a slot lies beyond the pool."""
    kn, vn = _bits(k_new), _bits(v_new)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, bs, h_kv, d = k_cache.shape
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous
    return (lib or _lib()).oracle_append_fp8(
        _ptr(k_cache), _ptr(v_cache), _ptr(kn), _ptr(vn), _ptr(sm), int(sm.shape[0]), nb, bs,
        h_kv, d, float(k_scale), float(v_scale), DTYPE_CODES[dtype])


def decode_attention_fp8(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                         block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
                         k_scale: float, v_scale: float, dtype: str,
                         lib: ctypes.CDLL = None) -> np.ndarray:
    """Decode attention over E4M3 caches (uint8 [num_blocks, bs, H_kv, d]) whose
    values are code * k_scale and code * v_scale; q uint16 of ``dtype``.
    Otherwise as ``decode_attention``.  Returns float64 [B, H_q, d]."""
    q = _bits(q)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    num_seqs, h_q, d = q.shape
    num_blocks, bs, h_kv, d2 = kc.shape
    if d2 != d or vc.shape != kc.shape or cl.shape != (num_seqs,):
        raise ValueError("inconsistent shapes")
    out = np.empty((num_seqs, h_q, d), dtype=np.float64)
    rc = (lib or _lib()).oracle_decode_attention_fp8(
        _ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), int(bt.shape[1]), _ptr(cl), num_seqs,
        num_blocks, bs, h_q, h_kv, d, float(scale), float(k_scale), float(v_scale),
        DTYPE_CODES[dtype])
    if rc == -1:
        raise ValueError("invalid arguments")
    if rc == -2:
        raise ValueError("block id out of range")
    return out


def decode_attention_np(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                        block_tables: np.ndarray, context_lens: np.ndarray,
                        scale: float) -> np.ndarray:
    """The same definition with numpy on float64 inputs (small cases).

    q float64 [B, H_q, d]; caches float64 [num_blocks, bs, H_kv, d].
    """
    num_seqs, h_q, d = q.shape
    h_kv = k_cache.shape[2]
    group = h_q // h_kv
    out = np.zeros((num_seqs, h_q, d), dtype=np.float64)
    for b in range(num_seqs):
        n = int(context_lens[b])
        if n <= 0:
            continue
        for h in range(h_q):
            k, v = gather_kv(k_cache, v_cache, block_tables, n, b, h // group)
            s = scale * (k @ q[b, h])
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ v
    return out


# ---------------------------------------------------------------------------
# The pages' per-page decode and its combine
# ---------------------------------------------------------------------------

def segment_partials(q_row: np.ndarray, k: np.ndarray, v: np.ndarray,
                     boundaries: Sequence[int], scale: float
                     ) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Local attention on each segment [boundaries[i], boundaries[i+1]) of one head.

    Per segment: S = scale * q K^T, M = max S, L = sum exp(S - M),
    P = exp(S - M) / L, O = P V (inference.html, "Decode 阶段的 PageAttention").
    Returns (O [P, d], L [P], M [P]).  An empty segment gets O = 0, L = 0,
    M = -inf.
    """
    outs, ls, ms = [], [], []
    for lo, hi in zip(boundaries[:-1], boundaries[1:]):
        if hi <= lo:
            outs.append(np.zeros(v.shape[1]))
            ls.append(0.0)
            ms.append(-math.inf)
            continue
        s = scale * (k[lo:hi] @ q_row)
        m = s.max()
        e = np.exp(s - m)
        l_sum = e.sum()
        outs.append((e / l_sum) @ v[lo:hi])
        ls.append(l_sum)
        ms.append(m)
    return np.array(outs), np.array(ls), np.array(ms)


def combine_result(o: np.ndarray, l_sum: np.ndarray, m: np.ndarray) -> np.ndarray:
    """Online-softmax combine of per-segment partials (inference.html, combine_result).

    M* = max_i M_i;  L* = sum_i exp(M_i - M*) L_i;
    O  = sum_i exp(M_i - M*) (L_i / L*) O_i.
    Segments with M_i = -inf (empty) carry weight 0; if every segment is empty
    the result is 0.
    """
    m_star = np.max(m)
    if not np.isfinite(m_star):
        return np.zeros(o.shape[1])
    scale_i = np.where(np.isfinite(m), np.exp(np.where(np.isfinite(m), m, 0.0) - m_star), 0.0)
    l_star = np.sum(scale_i * l_sum)
    return np.sum((scale_i * (l_sum / l_star))[:, None] * o, axis=0)


def decode_attention_pagewise(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                              block_tables: np.ndarray, context_lens: np.ndarray,
                              scale: float) -> np.ndarray:
    """The pages' method end to end: dispatch q to every page, attend locally, combine.

    Each page of the sequence (block_size tokens, the last one possibly partial)
    is one segment.  float64 inputs as in ``decode_attention_np``.
    """
    num_seqs, h_q, d = q.shape
    bs = k_cache.shape[1]
    group = h_q // k_cache.shape[2]
    out = np.zeros((num_seqs, h_q, d))
    for b in range(num_seqs):
        n = int(context_lens[b])
        if n <= 0:
            continue
        bounds = list(range(0, n, bs)) + [n]
        for h in range(h_q):
            k, v = gather_kv(k_cache, v_cache, block_tables, n, b, h // group)
            o, l_sum, m = segment_partials(q[b, h], k, v, bounds, scale)
            out[b, h] = combine_result(o, l_sum, m)
    return out


# ---------------------------------------------------------------------------
# Log-sum-exp merge of split partials
# ---------------------------------------------------------------------------

def merge_lse(partial_o: np.ndarray, partial_lse: np.ndarray) -> np.ndarray:
    """Merge normalised split partials stored with their log-sum-exp.

    partial_o [..., P, d] (each O_p already divided by its own sum),
    partial_lse [..., P] with lse_p = M_p + ln L_p (-inf for an empty split).
    Because exp(M_p - M*) L_p = exp(lse_p - M*), this is the combine rule of
    inference.html combine_result:  lse* = max_p lse_p,  w_p = exp(lse_p - lse*),
    O = sum_p w_p O_p / sum_p w_p.  Rows whose splits are all empty give 0.
    """
    po = np.asarray(partial_o, dtype=np.float64)
    pl = np.asarray(partial_lse, dtype=np.float64)
    lse_star = np.max(pl, axis=-1, keepdims=True)
    finite_star = np.isfinite(lse_star)
    safe_star = np.where(finite_star, lse_star, 0.0)
    w = np.where(np.isfinite(pl), np.exp(np.where(np.isfinite(pl), pl, 0.0) - safe_star), 0.0)
    den = w.sum(axis=-1, keepdims=True)
    num = (w[..., None] * po).sum(axis=-2)
    out = np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)
    return out
