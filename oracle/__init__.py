"""Oracle for paged-KV decode attention — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU implementation (fp64) of what the CUDA
library computes: the append (scatter through ``slot_mapping``), the gather
through the block table, decode attention ``softmax(q K^T * scale) V`` with
GQA, causal multi-query attention (several new query tokens per sequence), the
E4M3 (FP8) cache codes with their quantising append and decode attention,
the pages' per-page partials and their online-softmax combine, and the
log-sum-exp merge of split partials.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import or run anything in this package.  It shares no code with the
CUDA library (``paged_kv_cache_164_gb300``) and never imports it; the product
path never imports this package.

Every function is pinned by CPU tests to things other than itself: a dense
contiguous attention computed with library routines, hand-derived closed
forms, brute force on tiny inputs, invariants (block permutation, split and
merge), and the pages' worked KV-size examples.
"""
from .reference import (  # noqa: F401
    DTYPE_CODES,
    append,
    combine_result,
    append_fp8,
    decode_attention,
    decode_attention_fp8,
    decode_e4m3,
    decode_attention_np,
    decode_attention_pagewise,
    decode_values,
    encode_e4m3,
    gather_kv,
    kv_cache_bytes,
    merge_lse,
    multi_query_attention,
    num_threads,
    segment_partials,
)
