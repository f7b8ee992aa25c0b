"""Head-major caches ([num_blocks][H_kv][block_size][d]) and larger pages.

A head-major cache here is a workload's token-major cache with its values
permuted.  Append and gather must give bit-identical results in either
layout; decode (plain, fused, shared prefix, multi-query) on the head-major
copy must match the oracle run on the token-major cache.
"""
import pytest
import torch

import oracle
import paged_kv_cache_164_gb300 as pkv
from helpers import assert_attention_close, oracle_after_append
from workloads import bits, make_append_case, make_queries, make_workload, to_head_major

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_append_head_major_is_the_permuted_token_major_append(bs, dtype):
    c = make_append_case(300, 24, bs, 8, 128, dtype, seed=bs + len(dtype), device="cuda")
    kh, vh = to_head_major(c["k_cache"]), to_head_major(c["v_cache"])
    pkv.append(c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], c["slot_mapping"])
    flag = pkv.new_error_flag("cuda")
    pkv.append(c["k_new"], c["v_new"], kh, vh, c["slot_mapping"], err_flag=flag, layout="hnd")
    assert pkv.check_error(flag) == 0
    assert torch.equal(kh.view(torch.int16), to_head_major(c["k_cache"]).view(torch.int16))
    assert torch.equal(vh.view(torch.int16), to_head_major(c["v_cache"]).view(torch.int16))


@pytest.mark.parametrize("bs", [16, 64, 128])
def test_gather_head_major_equals_token_major(bs):
    w = make_workload("c3", device="cuda", num_seqs=5, block_size=bs, lengths=("uniform", 30, 900),
                      max_len_cap=1024, seed=81)
    k1, v1 = pkv.gather(w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.max_context_len)
    k2, v2 = pkv.gather(to_head_major(w.k_cache), to_head_major(w.v_cache), w.block_tables,
                        w.context_lens, w.max_context_len, layout="hnd")
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))


DECODE = {
    "gqa8_bf16_bs64": dict(name="c3", num_seqs=6, block_size=64, lengths=("uniform", 60, 2000),
                           max_len_cap=2048, seed=82),
    "gqa8_bf16_bs128": dict(name="c3", num_seqs=5, block_size=128, lengths=("uniform", 100, 2000),
                            max_len_cap=2048, seed=83),
    "mha_fp16_bs16": dict(name="c2", num_seqs=4, num_q_heads=8, num_kv_heads=8,
                          lengths=("uniform", 10, 900), max_len_cap=960, seed=84),
    "gqa4_d64_bs32": dict(name="c5_bs32", num_seqs=6, head_dim=64, shared_prefix_groups=0,
                          lengths=("uniform", 20, 700), max_len_cap=768, seed=85),
}


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("key", sorted(DECODE))
def test_decode_on_head_major_cache(key, splits):
    case = dict(DECODE[key])
    w = make_workload(case.pop("name"), device="cuda", poison=True, **case)
    expect, kc, vc = oracle_after_append(w)
    kh, vh = to_head_major(w.k_cache), to_head_major(w.v_cache)
    pkv.append(w.k_new, w.v_new, kh, vh, w.slot_mapping, layout="hnd")
    flag = pkv.new_error_flag("cuda")
    out = pkv.decode_attention(w.q, kh, vh, w.block_tables, w.context_lens, w.max_context_len,
                               scale=w.scale, num_splits=splits, err_flag=flag, layout="hnd")
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, expect, f"{key} splits={splits}")


@pytest.mark.parametrize("key", ["gqa8_bf16_bs128", "mha_fp16_bs16"])
def test_fused_append_decode_on_head_major_cache(key):
    case = dict(DECODE[key])
    w = make_workload(case.pop("name"), device="cuda", poison=True, **case)
    expect, _, _ = oracle_after_append(w)
    kh, vh = to_head_major(w.k_cache), to_head_major(w.v_cache)
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = pkv.append_decode_attention(w.q, w.k_new, w.v_new, kh, vh, w.block_tables,
                                      w.context_lens, w.max_context_len, scale=w.scale,
                                      layout="hnd")
    assert torch.equal(kh.view(torch.int16), to_head_major(w.k_cache).view(torch.int16))
    assert torch.equal(vh.view(torch.int16), to_head_major(w.v_cache).view(torch.int16))
    assert_attention_close(out, expect, key)


def test_shared_prefix_on_head_major_cache_with_64_token_pages():
    w = make_workload("c5", device="cuda", poison=True, num_seqs=16, block_size=64,
                      lengths=("prefix_lognormal", 256, 300, 1.0, 1500), max_len_cap=1536,
                      shared_prefix_groups=2, seed=86)
    expect, _, _ = oracle_after_append(w)
    kh, vh = to_head_major(w.k_cache), to_head_major(w.v_cache)
    pkv.append(w.k_new, w.v_new, kh, vh, w.slot_mapping, layout="hnd")
    flag = pkv.new_error_flag("cuda")
    out = pkv.decode_attention_prefix_shared(
        w.q, kh, vh, w.block_tables, w.context_lens, w.max_context_len, w.group_start,
        w.group_prefix_len, w.max_group_size, w.max_prefix_len, scale=w.scale, err_flag=flag,
        layout="hnd")
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, expect, "shared prefix, head-major, bs 64")


@pytest.mark.parametrize("q_len", [6, 2])  # 48 rows: tensor-core kernel; 16: decode kernel
def test_multi_query_on_head_major_cache_with_128_token_pages(q_len):
    case = dict(DECODE["gqa8_bf16_bs128"])
    w = make_workload(case.pop("name"), device="cuda", poison=True, **case)
    _, kc, vc = oracle_after_append(w)
    kh, vh = to_head_major(w.k_cache), to_head_major(w.v_cache)
    pkv.append(w.k_new, w.v_new, kh, vh, w.slot_mapping, layout="hnd")
    q = make_queries(w, q_len, seed=15)
    flag = pkv.new_error_flag("cuda")
    out = pkv.multi_query_attention(q, kh, vh, w.block_tables, w.context_lens, w.max_context_len,
                                    scale=w.scale, err_flag=flag, layout="hnd")
    assert pkv.check_error(flag) == 0
    expect = oracle.multi_query_attention(bits(q), kc, vc, w.block_tables.cpu().numpy(),
                                          w.context_lens.cpu().numpy(), w.scale, w.spec.dtype)
    assert_attention_close(out, expect, "multi-query, head-major, bs 128")
