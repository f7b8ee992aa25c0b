"""The C-ABI library loads, exports every declared symbol, and validates on the host (CPU)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_164_gb300 as pkv
from paged_kv_cache_164_gb300 import build as pkv_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"pkv_append", "pkv_decode_attention", "pkv_merge"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert pkv.status_string(code) != "unknown status"
    assert pkv.status_string(99) == "unknown status"
    assert lib.pkv_max_group_size() == 16


NULL = ctypes.c_void_p(0)


def test_append_rejects_bad_arguments_without_launching(lib):
    ok_args = dict(nt=4, nb=8, bs=16, h=2, d=64, dt=0)
    # null pointers
    assert lib.pkv_append(NULL, NULL, NULL, NULL, NULL, 4, 8, 16, 2, 64, 0, NULL, NULL) == 1
    # negative sizes, bad dtype
    assert lib.pkv_append(NULL, NULL, NULL, NULL, NULL, -1, 8, 16, 2, 64, 0, NULL, NULL) == 1
    assert lib.pkv_append(NULL, NULL, NULL, NULL, NULL, 4, 8, 16, 2, 64, 7, NULL, NULL) == 1
    # zero tokens is a no-op
    assert lib.pkv_append(NULL, NULL, NULL, NULL, NULL, 0, 8, 16, 2, 64, 0, NULL, NULL) == 0
    assert ok_args


def _decode(lib, **kw):
    a = dict(out=NULL, q=NULL, k=NULL, v=NULL, bt=NULL, mb=4, cl=NULL, mcl=64, B=2, nb=8, bs=16,
             hq=4, hkv=2, d=64, scale=0.125, splits=0, ws=NULL, wsb=0, dt=0, err=NULL,
             stream=NULL)
    a.update(kw)
    return lib.pkv_decode_attention(a["out"], a["q"], a["k"], a["v"], a["bt"], a["mb"], a["cl"],
                                    a["mcl"], a["B"], a["nb"], a["bs"], a["hq"], a["hkv"],
                                    a["d"], a["scale"], a["splits"], a["ws"], a["wsb"], a["dt"],
                                    a["err"], a["stream"])


def test_decode_rejects_bad_arguments_without_launching(lib):
    assert _decode(lib) == 1                      # null pointers
    assert _decode(lib, hq=5, hkv=2) == 1         # heads not a multiple
    assert _decode(lib, d=96) == 2                # unsupported head_dim
    assert _decode(lib, bs=8) == 2                # unsupported block_size
    assert _decode(lib, hq=34, hkv=2) == 2        # group of 17 > 16
    assert _decode(lib, splits=-1) == 1
    assert _decode(lib, splits=5000) == 1
    assert _decode(lib, dt=3) == 1
    assert _decode(lib, scale=float("nan")) == 1
    assert _decode(lib, B=0) == 0                 # empty batch is a no-op
    assert _decode(lib, dt=0x200) == 1            # an unknown flag in the dtype argument
    assert _decode(lib, dt=pkv.LAYOUT_HND, B=0) == 0   # the head-major flag is accepted
    assert _decode(lib, bs=128, d=96) == 2        # 128-token pages are fine, head_dim 96 is not


def test_workspace_size_rejects_bad_arguments(lib):
    assert lib.pkv_decode_workspace_size(2, 5, 2, 64, 16, 64, 0) == pkv.SIZE_MAX
    assert lib.pkv_decode_workspace_size(2, 4, 2, 96, 16, 64, 1) == pkv.SIZE_MAX
    # an explicit single partition needs no workspace and no device query
    assert lib.pkv_decode_workspace_size(2, 4, 2, 64, 16, 64, 1) == 0
    assert lib.pkv_decode_num_splits(2, 4, 2, 64, 16, 64, 1) == 1
    assert lib.pkv_decode_num_splits(2, 4, 2, 64, 16, 64, 3) == 2   # 4 pages -> 2 chunks of 2
    assert lib.pkv_decode_num_splits(2, 4, 2, 64, 16, 64, 2000) == -1
    assert lib.pkv_decode_num_splits(2, 4, 2, 64, 16, 64, 8) == 4     # no more than the pages
    assert lib.pkv_decode_num_splits_fp8(2, 4, 2, 64, 16, 64, 3) == 2
    assert lib.pkv_decode_num_splits_fp8(2, 4, 2, 64, 16, 64, 2000) == -1
    parts = ctypes.c_int(0)
    assert lib.pkv_multi_query_plan(2, 0, 4, 2, 64, 16, 64, ctypes.byref(parts)) == -1  # q_len 0
    assert lib.pkv_multi_query_plan(2, 4, 4, 2, 96, 16, 64, None) == -1  # head_dim 96
    assert lib.pkv_multi_query_plan(2, 4, 5, 2, 64, 16, 64, None) == -1  # heads not a multiple


def _multi_query(lib, **kw):
    a = dict(out=NULL, q=NULL, k=NULL, v=NULL, bt=NULL, mb=4, cl=NULL, mcl=64, B=2, ql=3, nb=8,
             bs=16, hq=4, hkv=2, d=64, scale=0.125, ws=NULL, wsb=0, dt=0, err=NULL, stream=NULL)
    a.update(kw)
    return lib.pkv_multi_query_attention(a["out"], a["q"], a["k"], a["v"], a["bt"], a["mb"],
                                         a["cl"], a["mcl"], a["B"], a["ql"], a["nb"], a["bs"],
                                         a["hq"], a["hkv"], a["d"], a["scale"], a["ws"], a["wsb"],
                                         a["dt"], a["err"], a["stream"])


def test_append_decode_rejects_bad_arguments_without_launching(lib):
    f = lib.pkv_append_decode_attention
    # null pointers (including the new tokens), bad head_dim, empty batch
    assert f(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 4, NULL, 64, 2, 8, 16, 4, 2, 64, 0.125, 1,
             NULL, 0, 0, NULL, NULL) == 1
    assert f(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 4, NULL, 64, 2, 8, 16, 4, 2, 96, 0.125, 1,
             NULL, 0, 0, NULL, NULL) == 2
    assert f(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 4, NULL, 64, 0, 8, 16, 4, 2, 64, 0.125, 1,
             NULL, 0, 0, NULL, NULL) == 0


def test_multi_query_rejects_bad_arguments_without_launching(lib):
    assert _multi_query(lib) == 1                 # null pointers
    assert _multi_query(lib, ql=0) == 1           # no query tokens
    assert _multi_query(lib, hq=5, hkv=2) == 1    # heads not a multiple
    assert _multi_query(lib, d=96) == 2           # unsupported head_dim
    assert _multi_query(lib, bs=8) == 2           # unsupported block_size
    assert _multi_query(lib, dt=3) == 1
    assert _multi_query(lib, scale=float("inf")) == 1
    assert _multi_query(lib, B=0) == 0            # empty batch is a no-op
    assert lib.pkv_multi_query_workspace_size(2, 0, 4, 2, 64, 16, 64) == pkv.SIZE_MAX
    assert lib.pkv_multi_query_workspace_size(2, 3, 4, 2, 96, 16, 64) == pkv.SIZE_MAX


def test_merge_and_gather_reject_bad_arguments(lib):
    assert lib.pkv_merge(NULL, NULL, NULL, 2, 4, 3, 64, 0, NULL) == 1
    assert lib.pkv_merge(NULL, NULL, NULL, 2, 4, 0, 64, 0, NULL) == 1
    assert lib.pkv_gather(NULL, NULL, NULL, NULL, NULL, 4, NULL, 64, 2, 8, 16, 2, 64, 0, NULL,
                          NULL) == 1
    assert lib.pkv_check_error(NULL, NULL, None) == 1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    k = torch.zeros(4, 16, 2, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.append(k[:1, 0], k[:1, 0], k, k, torch.zeros(1, dtype=torch.int64))


def test_library_sources_allocate_no_device_memory():
    # The library allocates nothing on the device: the caller passes every
    # buffer (and the no-alloc entry point uses a static array).  No source of
    # the library names an allocating runtime or driver call.
    csrc = os.path.join(os.path.dirname(os.path.dirname(__file__)), "paged_kv_cache_164_gb300",
                        "csrc")
    banned = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cuMemAlloc\w*|cuMemFree\w*|"
                        r"cudaMallocAsync|cudaMemPool\w*|cuMemCreate)\b")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        assert not banned.search(text), f"{name} names {banned.search(text).group(0)}"


def _append_decode_fp8(lib, **kw):
    fake = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never dereferenced: the call rejects first
    a = dict(out=fake, q=fake, kn=fake, vn=fake, k=fake, v=fake, bt=fake, mb=4, cl=fake, mcl=64,
             B=2, nb=8, bs=16, hq=16, hkv=2, d=128, scale=0.088, ks=0.01, vs=0.02, splits=0,
             ws=NULL, wsb=0, dt=1, err=NULL, stream=NULL)
    a.update(kw)
    return lib.pkv_append_decode_attention_fp8(
        a["out"], a["q"], a["kn"], a["vn"], a["k"], a["v"], a["bt"], a["mb"], a["cl"], a["mcl"],
        a["B"], a["nb"], a["bs"], a["hq"], a["hkv"], a["d"], a["scale"], a["ks"], a["vs"],
        a["splits"], a["ws"], a["wsb"], a["dt"], a["err"], a["stream"])


def test_append_decode_fp8_rejects_bad_arguments_without_launching(lib):
    assert _append_decode_fp8(lib, kn=NULL) == 1          # the new tokens are required
    assert _append_decode_fp8(lib, vn=NULL) == 1
    assert _append_decode_fp8(lib, out=NULL) == 1
    assert _append_decode_fp8(lib, d=64, hq=4) == 2       # an E4M3 stage row holds 128 dims
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert _append_decode_fp8(lib, ks=bad) == 1       # scales positive and finite
        assert _append_decode_fp8(lib, vs=bad) == 1
    assert _append_decode_fp8(lib, dt=3) == 1             # fp16 or bf16 activations only
    assert _append_decode_fp8(lib, hq=5) == 1             # heads not a multiple of the KV heads
    assert _append_decode_fp8(lib, bs=8) == 2             # unsupported page size
    assert _append_decode_fp8(lib, B=0, kn=NULL, vn=NULL) == 0  # empty batch is a no-op
