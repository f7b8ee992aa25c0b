"""Causal multi-query attention (q_len new tokens per sequence) on the GPU vs the fp64 oracle.

The chunk's K/V are appended first (context_lens counts them); query token i of
a sequence with n cached tokens attends to positions 0 .. n - q_len + i.  The
oracle applies the decode-attention definition to every query token with its
own causal context.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_164_gb300 as pkv
from helpers import assert_attention_close
from workloads import bits, make_queries, make_workload

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_gqa2_fp16_d64": dict(name="c1", q_len=4),
    "spec_verify_gqa8_bf16": dict(name="c3", q_len=5, num_seqs=4, lengths=("uniform", 200, 700),
                                  max_len_cap=768, seed=61),
    "chunk64_gqa4_bf16_two_row_tiles": dict(name="c5", q_len=64, num_seqs=3,
                                            lengths=("uniform", 300, 1100), max_len_cap=1152,
                                            shared_prefix_groups=0, seed=62),
    "mha_fp16_d128_q16": dict(name="c2", q_len=16, num_seqs=3, num_q_heads=4, num_kv_heads=4,
                              lengths=("uniform", 40, 500), max_len_cap=512, seed=63),
    "gqa16_q8_full_tile": dict(name="c3", q_len=8, num_seqs=2, num_q_heads=32, num_kv_heads=2,
                               lengths=("uniform", 90, 300), max_len_cap=320, seed=64),
    "bs32_d64_q3": dict(name="c5_bs32", q_len=3, num_seqs=5, head_dim=64,
                        lengths=("uniform", 20, 400), max_len_cap=416, shared_prefix_groups=0,
                        seed=65),
    # 64 rows per (sequence, KV head) run the four-threads-per-row layout, 72
    # rows the two-threads-per-row one: both sides of the switch
    "gqa8_q8_rows64_long": dict(name="c3", q_len=8, num_seqs=3, lengths=("uniform", 1500, 2600),
                                max_len_cap=2688, seed=66),
    "gqa8_q9_rows72": dict(name="c3", q_len=9, num_seqs=3, lengths=("uniform", 60, 900),
                           max_len_cap=960, seed=67),
    # At most 32 (query token, head) rows per (sequence, KV head) run on the
    # decode kernel (rows as its columns): one and two 8-column groups, one and
    # two row blocks (CTAs) per (sequence, KV head), one partition (direct
    # output) and several (partials + merge); 33 rows are the tensor-core
    # kernel's again.
    "mha_q4_split_merge": dict(name="c2", q_len=4, num_seqs=3, num_q_heads=4, num_kv_heads=4,
                               lengths=("uniform", 1500, 4000), max_len_cap=4096, seed=68),
    "gqa8_q2_rows16": dict(name="c3", q_len=2, num_seqs=3, lengths=("uniform", 100, 1800),
                           max_len_cap=1856, seed=69),
    "gqa2_q8_fp16_d64_rows16": dict(name="c1", q_len=8),
    "mha_q17_rows17_two_blocks": dict(name="c2", q_len=17, num_seqs=2, num_q_heads=4,
                                      num_kv_heads=4, lengths=("uniform", 30, 400),
                                      max_len_cap=448, seed=70),
    "gqa8_q3_rows24": dict(name="c3", q_len=3, num_seqs=3, lengths=("uniform", 100, 1800),
                           max_len_cap=1856, seed=71),
    "gqa8_q4_rows32_split": dict(name="c3", q_len=4, num_seqs=2, lengths=("uniform", 2500, 4000),
                                 max_len_cap=4096, seed=72),
    "mha_q33_rows33": dict(name="c2", q_len=33, num_seqs=2, num_q_heads=4, num_kv_heads=4,
                           lengths=("uniform", 40, 400), max_len_cap=448, seed=73),
    "gqa4_d64_bs32_q6_rows24": dict(name="c5_bs32", q_len=6, num_seqs=4, head_dim=64,
                                    lengths=("uniform", 30, 2500), max_len_cap=2560,
                                    shared_prefix_groups=0, seed=74),
    # many ragged units (some shorter than one tile) at 32-token pages; long
    # contexts split into many partitions and merged; fp16 MHA with 20 rows
    "gqa8_q3_many_ragged_bs32": dict(name="c3", q_len=3, num_seqs=12, block_size=32,
                                     lengths=("uniform", 3, 3000), max_len_cap=3008, seed=75),
    "gqa8_q6_long_merged": dict(name="c3", q_len=6, num_seqs=2,
                                lengths=("uniform", 20000, 40000), max_len_cap=40000, seed=76),
    "mha_fp16_q20_rows20": dict(name="c2", q_len=20, num_seqs=3, num_q_heads=4, num_kv_heads=4,
                                lengths=("uniform", 20, 1500), max_len_cap=1536, seed=77),
}


def _make(key, **kw):
    case = dict(CASES[key])
    name = case.pop("name")
    q_len = case.pop("q_len")
    case.update(kw)
    w = make_workload(name, device="cuda", poison=True, **case)
    return w, q_len


def _appended(w):
    """Appends the workload's new tokens on the GPU and in host copies for the oracle."""
    flag = pkv.new_error_flag("cuda")
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, err_flag=flag)
    assert pkv.check_error(flag) == 0
    return bits(w.k_cache).copy(), bits(w.v_cache).copy()


def _expect(w, q, kc, vc, cl=None):
    cl = w.context_lens.cpu().numpy() if cl is None else cl
    return oracle.multi_query_attention(bits(q), kc, vc, w.block_tables.cpu().numpy(), cl,
                                        w.scale, w.spec.dtype)


@pytest.mark.parametrize("key", sorted(CASES))
def test_multi_query_matches_oracle(key):
    w, q_len = _make(key)
    kc, vc = _appended(w)
    q = make_queries(w, q_len, seed=11)
    flag = pkv.new_error_flag("cuda")
    out = pkv.multi_query_attention(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                    w.max_context_len, scale=w.scale, err_flag=flag)
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, _expect(w, q, kc, vc), key)


def test_one_query_token_matches_plain_decode():
    w, _ = _make("spec_verify_gqa8_bf16")
    _appended(w)
    q = make_queries(w, 1, seed=12)
    mq = pkv.multi_query_attention(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                   w.max_context_len, scale=w.scale)
    dec = pkv.decode_attention(q[:, 0].contiguous(), w.k_cache, w.v_cache, w.block_tables,
                               w.context_lens, w.max_context_len, scale=w.scale)
    assert torch.allclose(mq[:, 0].float(), dec.float(), atol=2e-3, rtol=1e-2)


def test_context_equal_to_chunk_and_shorter_than_chunk():
    w, q_len = _make("mha_fp16_d128_q16")
    kc, vc = _appended(w)
    q = make_queries(w, q_len, seed=13)
    cl = w.context_lens.clone()
    cl[0] = q_len          # the whole context is the chunk: token 0 sees only itself
    w.context_lens = cl
    flag = pkv.new_error_flag("cuda")
    out = pkv.multi_query_attention(q, w.k_cache, w.v_cache, w.block_tables, cl,
                                    w.max_context_len, scale=w.scale, err_flag=flag)
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, _expect(w, q, kc, vc, cl.cpu().numpy()), "context == q_len")
    # shorter than the chunk: flagged; rows with no visible position are zero
    cl2 = cl.clone()
    cl2[1] = q_len - 6
    out2 = pkv.multi_query_attention(q, w.k_cache, w.v_cache, w.block_tables, cl2,
                                     w.max_context_len, scale=w.scale, err_flag=flag)
    assert pkv.check_error(flag) & pkv.EFLAG_CONTEXT_LEN
    assert torch.count_nonzero(out2[1, :6]) == 0
    assert_attention_close(out2, _expect(w, q, kc, vc, cl2.cpu().numpy()), "context < q_len")


def test_full_size_llama70b_layer_speculative_verify_sampled():
    w = make_workload("c3", device="cuda")
    kc, vc = _appended(w)
    q_len = 8
    q = make_queries(w, q_len, seed=14)
    flag = pkv.new_error_flag("cuda")
    out = pkv.multi_query_attention(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                    w.max_context_len, scale=w.scale, err_flag=flag)
    assert pkv.check_error(flag) == 0
    seqs = np.array([0, 9, 21, 31])
    expect = oracle.multi_query_attention(bits(q)[seqs], kc, vc,
                                          w.block_tables.cpu().numpy()[seqs],
                                          w.context_lens.cpu().numpy()[seqs], w.scale,
                                          w.spec.dtype)
    assert_attention_close(out[torch.as_tensor(seqs, device="cuda")], expect, "c3 q_len 8")
    assert torch.isfinite(out).all()


def test_full_size_llama7b_layer_four_token_verify_sampled():
    """C2 (Llama-7B MHA layer, 64 sequences of 512-4096 tokens) with 4 query
    tokens per sequence: 4 rows per (sequence, KV head), the decode kernel's
    multi-query form, checked on sampled sequences."""
    w = make_workload("c2", device="cuda")
    kc, vc = _appended(w)
    q_len = 4
    q = make_queries(w, q_len, seed=16)
    flag = pkv.new_error_flag("cuda")
    out = pkv.multi_query_attention(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                    w.max_context_len, scale=w.scale, err_flag=flag)
    assert pkv.check_error(flag) == 0
    cl = w.context_lens.cpu().numpy()
    seqs = np.array([int(np.argmin(cl)), 17, 40, int(np.argmax(cl))])
    expect = oracle.multi_query_attention(bits(q)[seqs], kc, vc,
                                          w.block_tables.cpu().numpy()[seqs], cl[seqs], w.scale,
                                          w.spec.dtype)
    assert_attention_close(out[torch.as_tensor(seqs, device="cuda")], expect, "c2 q_len 4")
    assert torch.isfinite(out).all()


def test_rows_per_kv_head_choose_the_kernel():
    """Up to 32 (query token, head) rows per (sequence, KV head) go to the decode
    kernel (one CTA per 16 rows), planned like a decode; more go to the
    tensor-core kernel."""
    kernel, parts = pkv.multi_query_plan(64, 4, 32, 32, 128, 16, 4096)
    assert kernel == "decode"
    assert parts == pkv.decode_num_splits(64, 32, 32, 128, 16, 4096)
    assert pkv.multi_query_plan(32, 2, 64, 8, 128, 16, 4096)[0] == "decode"    # 16 rows
    assert pkv.multi_query_plan(32, 3, 64, 8, 128, 16, 4096)[0] == "decode"    # 24 rows
    assert pkv.multi_query_plan(32, 4, 64, 8, 128, 16, 4096)[0] == "decode"    # 32 rows
    assert pkv.multi_query_plan(32, 5, 64, 8, 128, 16, 4096)[0] == "tcgen05"   # 40 rows
    assert pkv.multi_query_plan(2, 33, 4, 4, 128, 16, 448)[0] == "tcgen05"     # 33 rows


@pytest.mark.parametrize("key", ["mha_q4_split_merge", "spec_verify_gqa8_bf16"])  # decode / tcgen05
def test_empty_context_gives_zero_rows_and_is_flagged(key):
    w, q_len = _make(key)
    kc, vc = _appended(w)
    q = make_queries(w, q_len, seed=17)
    cl = w.context_lens.clone()
    cl[0] = 0
    flag = pkv.new_error_flag("cuda")
    out = pkv.multi_query_attention(q, w.k_cache, w.v_cache, w.block_tables, cl,
                                    w.max_context_len, scale=w.scale, err_flag=flag)
    assert pkv.check_error(flag) & pkv.EFLAG_CONTEXT_LEN
    assert torch.count_nonzero(out[0]) == 0
    assert_attention_close(out[1:], _expect(w, q, kc, vc, cl.cpu().numpy())[1:], key + " n=0")
