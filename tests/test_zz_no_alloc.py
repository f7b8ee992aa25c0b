"""The allocation-free decode entry point (GPU).

pkv_decode_attention_noalloc serves callers that cannot allocate device memory:
plain-C hosts with no device allocator of their own, plug-ins that must not
bypass their host runtime's memory pool, and decode loops that cannot afford
the device-wide synchronisation cudaMalloc / cudaFree may cause.  It keeps its
split-K scratch in a fixed array inside the library, shared by every call.

These tests call it through the C ABI on workloads that need scratch, twice in
a row (the second call finds the first call's leftovers in the shared array),
and require each output to agree with the workspace-taking entry point and
with the fp64 oracle, within the attention tolerance the other tests use.  The
second call must leave torch's allocator untouched and take no device memory.
This file sorts last so that a run stopping at its first failure has already
run every other test.
"""
import ctypes
import math

import pytest
import torch

import paged_kv_cache_164_gb300 as pkv
from paged_kv_cache_164_gb300 import build as pkv_build
from helpers import assert_attention_close, oracle_after_append
from workloads import make_workload

pytestmark = pytest.mark.gpu


def _args(w, out):
    s = w.spec
    P = ctypes.c_void_p
    return [P(out.data_ptr()), P(w.q.data_ptr()), P(w.k_cache.data_ptr()),
            P(w.v_cache.data_ptr()), P(w.block_tables.data_ptr()), w.block_tables.shape[1],
            P(w.context_lens.data_ptr()), w.max_context_len, s.num_seqs, w.num_blocks,
            s.block_size, s.num_q_heads, s.num_kv_heads, s.head_dim,
            ctypes.c_float(w.scale)]


def _workload(name):
    kw = dict(num_seqs=6, lengths=("uniform", 300, 2000), max_len_cap=2048)
    if name == "c5":
        kw = dict(num_seqs=8, lengths=("prefix_lognormal", 256, 400, 1.0, 2000),
                  max_len_cap=2048, shared_prefix_groups=2)
    return make_workload(name, device="cuda", poison=True, **kw)


@pytest.mark.parametrize("name,splits", [("c3", 4), ("c5", 0), ("c2", 3)])
def test_noalloc_matches_workspace_call_and_oracle_twice(name, splits):
    pkv_build.build()
    lib = pkv.load()
    w = _workload(name)
    expect, _, _ = oracle_after_append(w)
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    s = w.spec
    dtype_code = 1 if s.dtype == "bf16" else 0
    need = lib.pkv_decode_workspace_size(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                         s.block_size, w.max_context_len, splits)
    assert 0 < need <= pkv.NOALLOC_SCRATCH_BYTES   # the case really uses scratch
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    # the workspace-taking entry point, for comparison
    ref = torch.empty_like(w.q)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = lib.pkv_decode_attention(*_args(w, ref), splits, ctypes.c_void_p(ws.data_ptr()), need,
                                  dtype_code, None, stream)
    assert st == 0
    torch.cuda.synchronize()
    assert_attention_close(ref, expect, f"{name} workspace call")
    ref64 = ref.double().cpu().numpy()

    outs = [torch.full_like(w.q, float("nan")) for _ in range(2)]
    flag = pkv.new_error_flag("cuda")
    torch.cuda.synchronize()
    for call in range(2):
        if call == 1:
            # after the first call's set-up: nothing is allocated, by torch or otherwise
            torch.cuda.synchronize()
            torch_bytes = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved())
            free_before = torch.cuda.mem_get_info()[0]
        st = lib.pkv_decode_attention_noalloc(*_args(w, outs[call]), splits, dtype_code,
                                              ctypes.c_void_p(flag.data_ptr()), stream)
        assert st == 0, pkv.status_string(st)
        assert pkv.check_error(flag) == 0
        if call == 1:
            assert (torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == torch_bytes
            assert torch.cuda.mem_get_info()[0] >= free_before
        assert_attention_close(outs[call], ref64, f"{name} no-alloc call {call + 1} vs workspace")
        assert_attention_close(outs[call], expect, f"{name} no-alloc call {call + 1} vs oracle")


def test_noalloc_python_binding():
    pkv_build.build()
    w = _workload("c3")
    expect, _, _ = oracle_after_append(w)
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = torch.empty_like(w.q)
    flag = pkv.new_error_flag("cuda")
    pkv.decode_attention_noalloc(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                 w.max_context_len, out, scale=w.scale, num_splits=5,
                                 err_flag=flag)
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, expect, "no-alloc through the binding")


def test_noalloc_rejects_plans_beyond_its_scratch():
    pkv_build.build()
    lib = pkv.load()
    w = make_workload("c3", num_seqs=64, lengths=("const", 4096), max_len_cap=4096,
                      with_values=False)
    s = w.spec
    need = lib.pkv_decode_workspace_size(64, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                         s.block_size, 4096, 64)
    assert need > pkv.NOALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = P(dummy.data_ptr())
    st = lib.pkv_decode_attention_noalloc(p, p, p, p, p, 256, p, 4096, 64, 8192, s.block_size,
                                          s.num_q_heads, s.num_kv_heads, s.head_dim,
                                          ctypes.c_float(1 / math.sqrt(128)), 64, 1, None,
                                          P(torch.cuda.current_stream().cuda_stream))
    assert st == 3   # PKV_ERR_WORKSPACE, nothing launched
