"""Decode attention on the GPU against the fp64 oracle.

Small cases (the oracle finishes in seconds) are compared element by element for
every split count; the full-size workloads, in the launch configuration the
benchmark uses (automatic splits), are compared on sampled sequences.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_164_gb300 as pkv
from helpers import assert_attention_close, oracle_after_append
from workloads import bits, make_workload

pytestmark = pytest.mark.gpu

SMALL = {
    "c1": dict(name="c1"),
    "mha_ragged": dict(name="c2", num_seqs=6, lengths=("uniform", 1, 700), max_len_cap=704),
    "gqa8_bf16": dict(name="c3", num_seqs=3, lengths=("uniform", 200, 1500), max_len_cap=1536,
                      pool="free_list", pool_slack=0.2),
    "gqa4_prefix_bs32": dict(name="c5_bs32", num_seqs=8,
                             lengths=("prefix_lognormal", 128, 200, 1.0, 1200), max_len_cap=1280,
                             shared_prefix_groups=2),
    "gqa4_prefix_bs16": dict(name="c5", num_seqs=8,
                             lengths=("prefix_lognormal", 128, 200, 1.0, 1200), max_len_cap=1280,
                             shared_prefix_groups=4),
    "gqa3_d64_fp16": dict(name="c2", num_seqs=4, num_q_heads=6, num_kv_heads=2, head_dim=64,
                          lengths=("uniform", 30, 300), max_len_cap=320, seed=21),
    "gqa16_bf16": dict(name="c3", num_seqs=2, num_q_heads=32, num_kv_heads=2, head_dim=128,
                       lengths=("uniform", 100, 400), max_len_cap=400, pool="free_list", seed=31),
}


def _make(key, device="cuda", **kw):
    case = dict(SMALL[key])
    name = case.pop("name")
    case.update(kw)
    return make_workload(name, device=device, **case)


def _run(w, num_splits=0, flag=None):
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, err_flag=flag)
    return pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                w.max_context_len, scale=w.scale, num_splits=num_splits,
                                err_flag=flag)


@pytest.mark.parametrize("key", sorted(SMALL))
@pytest.mark.parametrize("splits", [0, 1, 2, 4, 8])
def test_small_cases_all_splits(key, splits):
    w = _make(key, poison=True)
    expect, _, _ = oracle_after_append(w)
    flag = pkv.new_error_flag("cuda")
    out = _run(w, splits, flag)
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, expect, f"{key} splits={splits}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("key", ["mha_ragged", "gqa8_bf16", "gqa4_prefix_bs32"])
def test_both_dtypes(key, dtype):
    w = _make(key, dtype=dtype, poison=True)
    expect, _, _ = oracle_after_append(w)
    assert_attention_close(_run(w), expect, f"{key} {dtype}")


@pytest.mark.parametrize("n", [1, 2, 15, 16, 17, 31, 32, 33, 64, 65])
@pytest.mark.parametrize("bs", [16, 32])
def test_edge_lengths(n, bs):
    w = make_workload("c3", num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=64,
                      block_size=bs, lengths=("fixed", (n, max(1, n - 1), n + 1)),
                      max_len_cap=n + 1, pool="free_list", pool_slack=0.5, seed=n * 7 + bs,
                      device="cuda", poison=True)
    expect, _, _ = oracle_after_append(w)
    for splits in (0, 1, 3):
        assert_attention_close(_run(w, splits), expect, f"n={n} bs={bs} splits={splits}")


@pytest.mark.parametrize("group", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("d", [64, 128])
def test_group_sizes_and_head_dims(group, d):
    w = make_workload("c3", num_seqs=3, num_q_heads=2 * group, num_kv_heads=2, head_dim=d,
                      lengths=("uniform", 50, 600), max_len_cap=640, pool="free_list",
                      pool_slack=0.1, seed=group * 100 + d, device="cuda", poison=True)
    expect, _, _ = oracle_after_append(w)
    assert_attention_close(_run(w), expect, f"G={group} d={d}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("group", [8, 16])
@pytest.mark.parametrize("rise", [0.075, 0.117, 0.225, -0.075])
def test_scores_rising_across_stages(rise, group, dtype):
    """Scores that climb (or fall) steadily along the context by about `rise`
    (base 2) per token.  A consumer warp of the decode kernel takes every fourth
    16-token stage, so its consecutive stages lie 64 tokens apart: 0.117 raises
    the maximum between them by ~7.5, just under the 2^8 the running softmax
    reference tolerates (kept for one step with exponentials up to ~2^7.5, then
    moved), 0.075 by ~4.8 (kept, then moved, with exponentials up to ~2^4.8),
    0.225 by ~14.4 (moved every time); the partitions of each split count start
    their own.  K is nonzero in dim 0 only
    and the ramp is centred on the context, so every score is one exact product
    of at most ~80 in magnitude and the comparison measures the softmax, not
    fp32 summation of large logits."""
    lens = (600, 333)
    w = make_workload("c3", num_seqs=2, num_q_heads=2 * group, num_kv_heads=2, head_dim=128,
                      dtype=dtype, lengths=("fixed", lens), max_len_cap=608,
                      pool="free_list", pool_slack=0.1, seed=7 + group, device="cuda",
                      poison=True)
    bs = w.spec.block_size
    # head h's base-2 score of token t: rise * (1 + h / 256) * (t - n / 2)
    h = torch.arange(w.q.shape[1], device="cuda", dtype=torch.float32)
    w.q[:, :, 0] = (1.0 + h / 256.0)[None, :].to(w.q.dtype)
    unit = 1.0 / (w.scale * math.log2(math.e))
    for b, n in enumerate(lens):
        t = torch.arange(n, device="cuda")
        kv = torch.zeros(n, w.k_cache.shape[2], w.k_cache.shape[3], device="cuda")
        kv[:, :, 0] = (rise * (t.float() - n / 2) * unit)[:, None]
        blk = w.block_tables[b, t // bs].long()
        w.k_cache[blk[:-1], (t % bs)[:-1]] = kv[:-1].to(w.k_cache.dtype)
        w.k_new[b] = kv[-1].to(w.k_new.dtype)
    expect, _, _ = oracle_after_append(w)
    for splits in (0, 1, 3):
        assert_attention_close(_run(w, splits), expect,
                               f"rise={rise} G={group} {dtype} splits={splits}")


def test_context_len_zero_gives_zeros():
    w = _make("mha_ragged")
    expect, _, _ = oracle_after_append(w)
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    cl = w.context_lens.clone()
    cl[2] = 0
    for splits in (0, 1, 4):
        out = pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, cl,
                                   w.max_context_len, scale=w.scale, num_splits=splits)
        assert torch.all(out[2] == 0)
        keep = [0, 1, 3, 4, 5]
        assert_attention_close(out[keep], expect[keep], f"zero-len splits={splits}")


def test_last_pool_block_and_block_permutation():
    w = _make("gqa8_bf16")
    # move one sequence's first page to the last pool block
    bt = w.block_tables.clone()
    last = w.num_blocks - 1
    src = int(bt[0, 0])
    w.k_cache[[src, last]] = w.k_cache[[last, src]]
    w.v_cache[[src, last]] = w.v_cache[[last, src]]
    bt[bt == src] = -7
    bt[bt == last] = src
    bt[bt == -7] = last
    w.block_tables = bt
    bs = w.spec.block_size
    blk, off = w.slot_mapping // bs, w.slot_mapping % bs
    blk = torch.where(blk == src, last, torch.where(blk == last, src, blk))
    w.slot_mapping = blk * bs + off
    assert int(w.block_tables[0, 0]) == last
    expect, _, _ = oracle_after_append(w)
    assert_attention_close(_run(w), expect, "last block")


def test_deterministic():
    w = _make("gqa4_prefix_bs16")
    a = _run(w, 4).clone()
    b = _run(w, 4).clone()
    assert torch.equal(a, b)


def test_non_default_stream():
    w = _make("gqa8_bf16")
    expect, _, _ = oracle_after_append(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = _run(w, 0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert_attention_close(out, expect, "side stream")


# ------------------------------------------------------------------ full-size workloads

FULL = {"c1": None, "c2": 64, "c3": 32, "c4": 2, "c5": 24, "c5_bs32": 24}


@pytest.mark.parametrize("name", sorted(FULL))
def test_full_size_sampled(name):
    w = make_workload(name, device="cuda")
    flag = pkv.new_error_flag("cuda")
    out = _run(w, 0, flag)
    assert pkv.check_error(flag) == 0
    n_sample = FULL[name]
    b = w.spec.num_seqs
    if n_sample is None or n_sample >= b:
        seqs = np.arange(b)
    else:
        rng = np.random.default_rng(1234)
        seqs = np.sort(rng.choice(b, size=n_sample, replace=False))
    expect, _, _ = oracle_after_append(w, seqs)
    assert_attention_close(out[torch.as_tensor(seqs, device="cuda")], expect, name)
    # outputs of every sequence are finite and bounded by max |V| (a convex combination)
    assert torch.isfinite(out).all()
    assert float(out.abs().max()) <= float(w.v_cache.abs().max()) * (1 + 2**-7)


@pytest.mark.parametrize("name", ["c2", "c3", "c4"])
def test_full_size_fused_step_sampled(name):
    """The 16-bit step the benchmark times on the plain-path workloads: one fused
    append + decode launch with the automatic plan.  Every new token lands in
    its slot bit for bit; sampled outputs match the oracle."""
    w = make_workload(name, device="cuda")
    seqs = np.arange(w.spec.num_seqs)
    if FULL[name] < w.spec.num_seqs:
        seqs = np.sort(np.random.default_rng(4321).choice(w.spec.num_seqs, size=FULL[name],
                                                          replace=False))
    expect, kc_expect, vc_expect = oracle_after_append(w, seqs)
    flag = pkv.new_error_flag("cuda")
    out = pkv.append_decode_attention(w.q, w.k_new, w.v_new, w.k_cache, w.v_cache,
                                      w.block_tables, w.context_lens, w.max_context_len,
                                      scale=w.scale, err_flag=flag)
    assert pkv.check_error(flag) == 0
    h, d = w.spec.num_kv_heads, w.spec.head_dim
    slots = w.slot_mapping.cpu().numpy()
    for cache, host in ((w.k_cache, kc_expect), (w.v_cache, vc_expect)):
        got = bits(cache.view(-1, h, d)[w.slot_mapping])
        assert np.array_equal(got, host.reshape(-1, h, d)[slots])
    assert_attention_close(out[torch.as_tensor(seqs, device="cuda")], expect, f"{name} fused")
    assert torch.isfinite(out).all()


def test_long_context_plan_uses_at_least_four_partitions():
    w = make_workload("c4", with_values=False)
    s = w.spec
    assert pkv.decode_num_splits(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                 s.block_size, w.max_context_len, 0) >= 4


def test_direct_and_split_sequences_in_one_batch():
    # Short sequences fit one partition and are written by the decode kernel
    # directly; longer ones are split and merged.  Every explicit split count
    # and the automatic plan must leave both kinds correct.
    w = make_workload("c3", device="cuda", poison=True, num_seqs=4,
                      lengths=("uniform", 200, 700), max_len_cap=768, seed=61)
    expect, _, _ = oracle_after_append(w)
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    flag = pkv.new_error_flag("cuda")
    for splits in (0, 1, 2, 3, 4, 5, 8):
        out = pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                   w.max_context_len, scale=w.scale, num_splits=splits,
                                   err_flag=flag)
        assert pkv.check_error(flag) == 0
        assert_attention_close(out, expect, f"splits={splits}")
