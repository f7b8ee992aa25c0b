"""Seeded random small cases against the fp64 oracle (GPU).

Each case draws its shape at random from a fixed seed: batch, context lengths
(with page-edge lengths 1, bs, bs + 1, 2 bs - 1 and, for the plain decode, an
empty context), GQA group 1-16, head_dim 64/128, page size 16-128, layout,
element type, split count, and the entry point (plain decode, fused
append + decode, causal multi-query with q_len 2-12, shared-prefix decode).
Every output element is compared with the oracle run on the token-major cache;
the cache after the append (or the fused append) must equal the oracle's own
append bit for bit.  Unused cache slots are NaN, so a kernel reading a masked
token fails.  The seeds are fixed: a failure names a case that reproduces.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_164_gb300 as pkv
from helpers import assert_attention_close
from workloads import bits, make_queries, make_workload, to_head_major

NUM_CASES = 64
MODES = ("decode", "decode", "fused", "multi_query", "prefix_shared")


def draw_case(i: int) -> dict:
    rng = np.random.default_rng(7000 + i)
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32, 64, 128]))
    group = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    h_kv = int(rng.choice([1, 2, 4]))
    mode = MODES[i % len(MODES)]
    case = dict(index=i, mode=mode, head_dim=d, block_size=bs, num_kv_heads=h_kv,
                num_q_heads=h_kv * group, dtype=str(rng.choice(["fp16", "bf16"])),
                layout=str(rng.choice(["nhd", "hnd"])), splits=int(rng.choice([0, 0, 1, 2, 3, 5, 8])),
                q_len=int(rng.integers(2, 13)) if mode == "multi_query" else 1,
                zero_len=False, no_suffix=False)
    if mode == "prefix_shared":
        groups = int(rng.integers(1, 3))
        # sometimes groups of many members: several 128-row tiles of the prefix
        # kernel, members whose rows straddle two tiles when the group is 3 or 5
        per = int(rng.choice([1, 2, 3, 30, 44]))
        prefix = bs * int(rng.integers(1, max(2, 640 // bs)))
        cap = prefix + int(rng.integers(64, 1200))
        case.update(num_seqs=groups * per, shared_prefix_groups=groups,
                    lengths=("prefix_lognormal", prefix, int(rng.integers(16, 400)), 1.0, cap),
                    max_len_cap=cap,
                    # the first group's members end at the prefix: no suffix partitions
                    no_suffix=bool(rng.random() < 0.3))
        return case
    b = int(rng.integers(1, 6))
    edges = [1, bs, bs + 1, 2 * bs - 1, 15, 16, 17]
    lens = []
    for _ in range(b):
        n = int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(1, 1800))
        lens.append(max(n, case["q_len"]))
    case.update(num_seqs=b, lengths=("fixed", tuple(lens)),
                max_len_cap=int(max(lens) + rng.integers(0, 2 * bs)), shared_prefix_groups=0,
                zero_len=mode == "decode" and b > 1 and rng.random() < 0.3)
    return case


def _workload(case):
    keys = ("num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "block_size", "dtype",
            "lengths", "max_len_cap", "shared_prefix_groups")
    return make_workload("c3", device="cuda", poison=True, pool="free_list", pool_slack=0.3,
                         seed=9000 + case["index"], **{k: case[k] for k in keys})


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(NUM_CASES))
def test_random_case_matches_oracle(i):
    case = draw_case(i)
    w = _workload(case)
    what = f"fuzz case {i}: " + ", ".join(f"{k}={v}" for k, v in case.items() if k != "index")
    s = w.spec
    # the oracle's append into host copies of the token-major cache
    kc, vc = bits(w.k_cache).copy(), bits(w.v_cache).copy()
    assert oracle.append(kc, vc, bits(w.k_new), bits(w.v_new), w.slot_mapping.cpu().numpy()) == 0
    bt_h = w.block_tables.cpu().numpy()
    cl_h = w.context_lens.cpu().numpy().copy()
    cl = w.context_lens.clone()
    if case["zero_len"]:
        cl[0] = 0
        cl_h[0] = 0
    if case["no_suffix"]:
        g0, g1 = int(w.group_start[0]), int(w.group_start[1])
        cl[g0:g1] = int(w.group_prefix_len[0])
        cl_h[g0:g1] = int(w.group_prefix_len[0])
    layout = case["layout"]
    k_dev, v_dev = w.k_cache, w.v_cache
    if layout == "hnd":
        k_dev, v_dev = to_head_major(k_dev), to_head_major(v_dev)
    flag = pkv.new_error_flag("cuda")
    mode = case["mode"]

    if mode == "multi_query":
        q = make_queries(w, case["q_len"], seed=9100 + i)
        pkv.append(w.k_new, w.v_new, k_dev, v_dev, w.slot_mapping, err_flag=flag, layout=layout)
        out = pkv.multi_query_attention(q, k_dev, v_dev, w.block_tables, cl, w.max_context_len,
                                        scale=w.scale, err_flag=flag, layout=layout)
        expect = oracle.multi_query_attention(bits(q), kc, vc, bt_h, cl_h, w.scale, s.dtype)
    else:
        if mode == "fused":
            out = pkv.append_decode_attention(w.q, w.k_new, w.v_new, k_dev, v_dev, w.block_tables,
                                              cl, w.max_context_len, scale=w.scale,
                                              num_splits=case["splits"], err_flag=flag,
                                              layout=layout)
        else:
            pkv.append(w.k_new, w.v_new, k_dev, v_dev, w.slot_mapping, err_flag=flag,
                       layout=layout)
            if mode == "prefix_shared":
                out = pkv.decode_attention_prefix_shared(
                    w.q, k_dev, v_dev, w.block_tables, cl, w.max_context_len, w.group_start,
                    w.group_prefix_len, w.max_group_size, w.max_prefix_len, scale=w.scale,
                    err_flag=flag, layout=layout)
            else:
                out = pkv.decode_attention(w.q, k_dev, v_dev, w.block_tables, cl,
                                           w.max_context_len, scale=w.scale,
                                           num_splits=case["splits"], err_flag=flag,
                                           layout=layout)
        expect = oracle.decode_attention(bits(w.q), kc, vc, bt_h, cl_h, w.scale, s.dtype)
    assert pkv.check_error(flag) == 0, what
    if case["zero_len"]:
        assert torch.count_nonzero(out[0]) == 0, what
    assert_attention_close(out, expect, what)
    # the cache after the (fused) append equals the oracle's append, bit for bit
    # (NaN-poisoned slots included: nothing but the new tokens' slots is written)
    if layout == "hnd":
        k_dev = k_dev.permute(0, 2, 1, 3).contiguous()
        v_dev = v_dev.permute(0, 2, 1, 3).contiguous()
    assert np.array_equal(bits(k_dev), kc), what
    assert np.array_equal(bits(v_dev), vc), what


def test_cases_cover_the_space():
    """The fixed seeds reach every entry point, head_dim, page size, layout and
    element type, small and large GQA groups, page-edge and empty contexts (CPU)."""
    cases = [draw_case(i) for i in range(NUM_CASES)]
    for key, want in (("mode", {"decode", "fused", "multi_query", "prefix_shared"}),
                      ("head_dim", {64, 128}), ("block_size", {16, 32, 64, 128}),
                      ("layout", {"nhd", "hnd"}), ("dtype", {"fp16", "bf16"})):
        assert {c[key] for c in cases} == want, key
    assert {c["num_q_heads"] // c["num_kv_heads"] for c in cases} >= {1, 2, 8, 16}
    assert any(c["zero_len"] for c in cases)
    pre = [c for c in cases if c["mode"] == "prefix_shared"]
    assert any(c["no_suffix"] for c in pre)
    # a group of more than one 128-row tile whose GQA group does not divide 128
    per_group = [(c["num_seqs"] // c["shared_prefix_groups"], c["num_q_heads"] // c["num_kv_heads"])
                 for c in pre]
    assert any(m * g > 128 and 128 % g for m, g in per_group)
    assert any(m * g > 128 for m, g in per_group)
    lens = [n for c in cases if c["lengths"][0] == "fixed" for n in c["lengths"][1]]
    assert 1 in lens and 16 in lens and 17 in lens
