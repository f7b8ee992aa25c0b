"""Pins the oracle to things other than itself (CPU only).

Each test ties the fp64 oracle to an independent fact: the pages' printed
figures (tests/golden), a dense attention computed with torch library routines,
hand-derived closed forms, brute force on the tiny workload, or an invariant the
mathematics guarantees.  Together they catch a dropped scale, a wrong GQA index,
swapped block/offset arithmetic, K and V transposed, a missing max subtraction
or a wrong combine rule.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import bits, make_append_case, make_queries, make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.detach().cpu().to(torch.float64).numpy()


def _oracle(w, k_cache=None, v_cache=None, block_tables=None, context_lens=None, q=None):
    return oracle.decode_attention(
        bits(w.q if q is None else q), bits(w.k_cache if k_cache is None else k_cache),
        bits(w.v_cache if v_cache is None else v_cache),
        (w.block_tables if block_tables is None else block_tables).numpy(),
        (w.context_lens if context_lens is None else context_lens).numpy(), w.scale,
        w.spec.dtype)


def _dense_torch(w):
    """Dense attention with torch library routines: pages concatenated by reshape."""
    bs = w.spec.block_size
    group = w.spec.num_q_heads // w.spec.num_kv_heads
    q = w.q.to(torch.float64)
    kc = w.k_cache.to(torch.float64)
    vc = w.v_cache.to(torch.float64)
    out = torch.zeros_like(q)
    for b in range(w.spec.num_seqs):
        n = int(w.context_lens[b])
        if n == 0:
            continue
        npages = (n + bs - 1) // bs
        pages = w.block_tables[b, :npages].long()
        k = kc[pages].reshape(npages * bs, w.spec.num_kv_heads, -1)[:n]
        v = vc[pages].reshape(npages * bs, w.spec.num_kv_heads, -1)[:n]
        k = k.repeat_interleave(group, dim=1).transpose(0, 1)  # [H_q, n, d]
        v = v.repeat_interleave(group, dim=1).transpose(0, 1)
        s = torch.einsum("hd,hnd->hn", q[b], k) * w.scale
        p = torch.softmax(s, dim=-1)
        out[b] = torch.einsum("hn,hnd->hd", p, v)
    return out.numpy()


SMALL_CASES = [
    dict(name="c1"),
    dict(name="c2", num_seqs=3, lengths=("uniform", 1, 200), max_len_cap=256),
    dict(name="c3", num_seqs=2, lengths=("uniform", 40, 300), max_len_cap=320, pool="free_list",
         pool_slack=0.5),
    dict(name="c5_bs32", num_seqs=8, lengths=("prefix_lognormal", 64, 40, 1.0, 400),
         max_len_cap=512, shared_prefix_groups=2),
    dict(name="c2", num_seqs=2, num_q_heads=6, num_kv_heads=3, head_dim=64,
         lengths=("fixed", (17, 33)), max_len_cap=48, seed=11),
]


def _make(case, **kw):
    case = dict(case)
    name = case.pop("name")
    case.update(kw)
    return make_workload(name, **case)


# --------------------------------------------------------------------------- decoders

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_value_decoders_match_library_conversion(dtype):
    raw = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode_values(raw, dtype)
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    ref = torch.from_numpy(raw.view(np.int16).copy()).view(tdt).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# --------------------------------------------------------------------------- KV size

def _golden_rows(kind):
    rows = []
    with open(os.path.join(GOLDEN, "kv_cache_size.txt")) as f:
        for line in f:
            parts = line.split()
            if parts and parts[0] == kind:
                rows.append(parts[1:])
    return rows


def test_kv_size_matches_pages_worked_examples():
    rows = _golden_rows("exact")
    assert len(rows) == 3
    for name, *nums in rows:
        L, H, d, S, B, e, value = map(int, nums)
        assert oracle.kv_cache_bytes(L, H, d, S, B, e) == value, name
    # the page's "0.5 MB per token" and "2 GB" read in binary units
    assert oracle.kv_cache_bytes(32, 32, 128, 1, 1, 2) == 2**19
    assert oracle.kv_cache_bytes(32, 32, 128, 4096, 1, 2) == 2 * 2**30


def test_kv_size_records_page_erratum():
    (name, *nums), = _golden_rows("erratum")
    L, H, d, S, B, e, printed = map(int, nums)
    formula = oracle.kv_cache_bytes(L, H, d, S, B, e)
    assert formula == 1_342_177_280 and formula != printed
    assert oracle.kv_cache_bytes(64, H, d, S, B, e) == printed


def test_kv_size_gqa_compression_ratios():
    rows = _golden_rows("ratio")
    assert len(rows) == 3
    for name, h_mha, h_var, ratio in rows:
        full = oracle.kv_cache_bytes(80, int(h_mha), 128, 4096, 1, 2)
        var = oracle.kv_cache_bytes(80, int(h_var), 128, 4096, 1, 2)
        assert full == int(ratio) * var, name


def test_kv_size_equals_allocated_cache_bytes():
    w = make_workload("c5", num_seqs=8, lengths=("prefix_lognormal", 64, 40, 1.0, 400),
                      max_len_cap=512, shared_prefix_groups=2)
    allocated = (w.k_cache.numel() * w.k_cache.element_size()
                 + w.v_cache.numel() * w.v_cache.element_size())
    slots = w.num_blocks * w.spec.block_size
    assert oracle.kv_cache_bytes(1, w.spec.num_kv_heads, w.spec.head_dim, slots, 1, 2) == allocated


# --------------------------------------------------------------------------- gather

def test_gather_follows_pages_block_table_example():
    table = {}
    with open(os.path.join(GOLDEN, "block_table_example.txt")) as f:
        for line in f:
            p = line.split()
            if not p or p[0].startswith("#"):
                continue
            if p[0] == "block_size":
                bs = int(p[1])
                continue
            table.setdefault(int(p[0]), {})[int(p[1])] = int(p[2])
    num_blocks, h_kv, d = 8, 1, 2
    # each slot stores its own (physical block, offset)
    cache = np.zeros((num_blocks, bs, h_kv, d), dtype=np.int32)
    cache[:, :, 0, 0] = np.arange(num_blocks)[:, None]
    cache[:, :, 0, 1] = np.arange(bs)[None, :]
    tables = np.full((2, 3), -1, dtype=np.int32)
    for req, m in table.items():
        for logical, phys in m.items():
            tables[req - 1, logical] = phys
    k, _ = oracle.gather_kv(cache, cache, tables, 3 * bs, 0, 0)
    expect_blocks = [5] * bs + [7] * bs + [2] * bs
    assert k[:, 0].tolist() == expect_blocks
    assert k[:, 1].tolist() == list(range(bs)) * 3
    k, _ = oracle.gather_kv(cache, cache, tables, 2 * bs - 3, 1, 0)
    assert k[:, 0].tolist() == [1] * bs + [3] * (bs - 3)
    # token 20 of request 1: logical block 1 -> physical 7, offset 4
    k, _ = oracle.gather_kv(cache, cache, tables, 21, 0, 0)
    assert tuple(k[20]) == (7, 4)


# --------------------------------------------------------------------------- definition

@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: c["name"] + str(c.get("num_seqs", "")))
def test_c_oracle_equals_dense_library_attention(case):
    w = _make(case)
    got = _oracle(w)
    dense = _dense_torch(w)
    np.testing.assert_allclose(got, dense, rtol=0, atol=1e-12)
    mine_np = oracle.decode_attention_np(_np(w.q), _np(w.k_cache), _np(w.v_cache),
                                         w.block_tables.numpy(), w.context_lens.numpy(), w.scale)
    np.testing.assert_allclose(got, mine_np, rtol=0, atol=1e-12)


def test_brute_force_tiny_workload():
    """Pure-Python loops (math.exp, no numpy) on the tiny workload."""
    w = make_workload("c1")
    q = w.q.to(torch.float64).tolist()
    kc = w.k_cache.to(torch.float64).tolist()
    vc = w.v_cache.to(torch.float64).tolist()
    bt = w.block_tables.tolist()
    bs, group = w.spec.block_size, w.spec.num_q_heads // w.spec.num_kv_heads
    got = _oracle(w)
    for b in range(w.spec.num_seqs):
        n = int(w.context_lens[b])
        for h in range(w.spec.num_q_heads):
            g = h // group
            s = []
            for t in range(n):
                kt = kc[bt[b][t // bs]][t % bs][g]
                s.append(w.scale * sum(a * c for a, c in zip(q[b][h], kt)))
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            for j in range(w.spec.head_dim):
                o = sum(e[t] * vc[bt[b][t // bs]][t % bs][g][j] for t in range(n)) / z
                assert abs(o - got[b, h, j]) < 1e-12


def _one_seq_case(n, d=64, seed=3, dtype="bf16", h_q=2, h_kv=1):
    return make_workload("c3", num_seqs=1, num_q_heads=h_q, num_kv_heads=h_kv, head_dim=d,
                         lengths=("fixed", (n,)), max_len_cap=max(n, 1), pool="free_list",
                         pool_slack=1.0, seed=seed, dtype=dtype)


def test_single_token_returns_its_value_exactly():
    w = _one_seq_case(1)
    got = _oracle(w)
    blk = int(w.block_tables[0, 0])
    v0 = w.v_cache[blk, 0, 0].to(torch.float64).numpy()
    assert np.array_equal(got[0, 0], v0) and np.array_equal(got[0, 1], v0)


def test_zero_query_gives_mean_of_values():
    w = _one_seq_case(45)
    q = torch.zeros_like(w.q)
    got = _oracle(w, q=q)
    _, v = oracle.gather_kv(_np(w.k_cache), _np(w.v_cache), w.block_tables.numpy(), 45, 0, 0)
    np.testing.assert_allclose(got[0, 0], v.mean(axis=0), rtol=0, atol=1e-14)


def test_two_tokens_closed_form():
    w = _one_seq_case(2, d=64, seed=5, dtype="fp16")
    k, v = oracle.gather_kv(_np(w.k_cache), _np(w.v_cache), w.block_tables.numpy(), 2, 0, 0)
    q = _np(w.q)[0, 0]
    s0, s1 = w.scale * q @ k[0], w.scale * q @ k[1]
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))  # noqa: E731
    expect = sig(s0 - s1) * v[0] + sig(s1 - s0) * v[1]
    np.testing.assert_allclose(_oracle(w)[0, 0], expect, rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value_and_large_scores_do_not_overflow():
    w = _one_seq_case(40, d=64, seed=7)
    k_cache = w.k_cache.clone()
    q = torch.zeros_like(w.q)
    q[0, :, 0] = 64.0
    k_cache[:, :, :, 0] = 1.0
    t_star = 29
    blk = int(w.block_tables[0, t_star // 16])
    k_cache[blk, t_star % 16, 0, 0] = 256.0  # score gap (256-1)*64/8 = 2040
    got = _oracle(w, k_cache=k_cache, q=q)
    v_star = w.v_cache[blk, t_star % 16, 0].to(torch.float64).numpy()
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got[0, 0], v_star, rtol=0, atol=1e-300)


def test_context_len_zero_gives_zero_row():
    w = _make(SMALL_CASES[1])
    cl = w.context_lens.clone()
    cl[1] = 0
    got = _oracle(w, context_lens=cl)
    assert np.all(got[1] == 0.0)
    full = _oracle(w)
    assert np.array_equal(got[0], full[0]) and np.array_equal(got[2], full[2])


def test_gqa_equals_mha_with_repeated_kv_heads():
    w = make_workload("c3", num_seqs=2, lengths=("fixed", (70, 33)), max_len_cap=80,
                      num_q_heads=8, num_kv_heads=2, head_dim=64, pool="free_list",
                      pool_slack=0.3)
    group = 4
    k_rep = w.k_cache.repeat_interleave(group, dim=2).contiguous()
    v_rep = w.v_cache.repeat_interleave(group, dim=2).contiguous()
    gqa = _oracle(w)
    mha = oracle.decode_attention(bits(w.q), bits(k_rep), bits(v_rep), w.block_tables.numpy(),
                                  w.context_lens.numpy(), w.scale, w.spec.dtype)
    assert np.array_equal(gqa, mha)


# --------------------------------------------------------------------------- invariants

def test_block_permutation_leaves_output_bit_identical():
    w = _make(SMALL_CASES[3])
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(w.num_blocks, generator=g)          # new position of each block
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt = w.block_tables.clone()
    used = bt >= 0
    bt[used] = perm[bt[used].long()].to(torch.int32)
    assert np.array_equal(_oracle(w), _oracle(w, k_cache=k2, v_cache=v2, block_tables=bt))


def test_unused_slots_and_table_entries_do_not_matter():
    w = _make(SMALL_CASES[1], poison=True)
    clean = _make(SMALL_CASES[1])
    # context excludes the new token's (poisoned) slot: attend to the cached tokens only
    cl = w.context_lens - 1
    got = _oracle(w, context_lens=cl)
    ref = _oracle(clean, context_lens=cl)
    assert np.all(np.isfinite(got)) and np.array_equal(got, ref)
    bt = w.block_tables.clone()
    bs = w.spec.block_size
    for b in range(bt.shape[0]):
        used = (int(cl[b]) + bs - 1) // bs
        bt[b, used:] = 10**6  # garbage beyond the context is never read
    assert np.array_equal(_oracle(w, context_lens=cl, block_tables=bt), got)


def test_out_of_range_block_id_is_reported():
    w = _make(SMALL_CASES[0])
    bt = w.block_tables.clone()
    bt[0, 1] = w.num_blocks
    with pytest.raises(ValueError):
        _oracle(w, block_tables=bt)


# --------------------------------------------------------------------------- split / merge

def test_pagewise_decode_and_combine_equal_single_pass():
    for case in SMALL_CASES:
        w = _make(case)
        args = (_np(w.q), _np(w.k_cache), _np(w.v_cache), w.block_tables.numpy(),
                w.context_lens.numpy(), w.scale)
        np.testing.assert_allclose(oracle.decode_attention_pagewise(*args), _oracle(w),
                                   rtol=0, atol=1e-13)


def test_random_splits_merge_to_single_pass():
    w = _make(SMALL_CASES[2])
    rng = np.random.default_rng(0)
    kc, vc = _np(w.k_cache), _np(w.v_cache)
    full = _oracle(w)
    group = w.spec.num_q_heads // w.spec.num_kv_heads
    for b in range(w.spec.num_seqs):
        n = int(w.context_lens[b])
        for h in range(w.spec.num_q_heads):
            k, v = oracle.gather_kv(kc, vc, w.block_tables.numpy(), n, b, h // group)
            cuts = sorted(rng.choice(np.arange(1, n), size=5, replace=False).tolist())
            bounds = [0] + cuts + [n]
            bounds.insert(2, bounds[2])  # an empty segment in the middle
            o, l_sum, m = oracle.segment_partials(_np(w.q)[b, h], k, v, bounds, w.scale)
            np.testing.assert_allclose(oracle.combine_result(o, l_sum, m), full[b, h],
                                       rtol=0, atol=1e-13)
            lse = np.where(np.isfinite(m), m + np.log(np.where(l_sum > 0, l_sum, 1.0)), -np.inf)
            np.testing.assert_allclose(oracle.merge_lse(o, lse), full[b, h], rtol=0, atol=1e-13)


def test_merge_lse_edge_cases():
    o = np.array([[1.0, 2.0], [3.0, 4.0]])
    # all splits empty -> 0
    assert np.array_equal(oracle.merge_lse(o, np.array([-np.inf, -np.inf])), [0.0, 0.0])
    # one empty split carries no weight
    assert np.array_equal(oracle.merge_lse(o, np.array([-np.inf, 0.3])), [3.0, 4.0])
    # equal lse -> plain mean; lse differing by ln 3 -> weights 3:1
    np.testing.assert_allclose(oracle.merge_lse(o, np.array([0.0, 0.0])), [2.0, 3.0])
    np.testing.assert_allclose(oracle.merge_lse(o, np.array([math.log(3.0), 0.0])),
                               [1.5, 2.5], rtol=1e-15)


# --------------------------------------------------------------------------- append

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_append_matches_independent_scatter(dtype):
    c = make_append_case(300, 40, 16, 4, 64, dtype, seed=5)
    kc, vc = bits(c["k_cache"]).copy(), bits(c["v_cache"]).copy()
    slots = c["slot_mapping"].numpy()
    assert oracle.append(kc, vc, bits(c["k_new"]), bits(c["v_new"]), slots) == 0
    ek, ev = bits(c["k_cache"]).copy(), bits(c["v_cache"]).copy()
    keep = slots >= 0
    ek.reshape(-1, 4, 64)[slots[keep]] = bits(c["k_new"])[keep]
    ev.reshape(-1, 4, 64)[slots[keep]] = bits(c["v_new"])[keep]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)
    untouched = np.ones(40 * 16, dtype=bool)
    untouched[slots[keep]] = False
    assert np.all(kc.reshape(-1, 4, 64)[untouched] == 0x7E5A)


def test_append_reports_slot_beyond_pool():
    c = make_append_case(10, 4, 16, 2, 64, "fp16", seed=6, pad_fraction=0.0)
    slots = c["slot_mapping"].numpy().copy()
    slots[3] = 4 * 16
    kc, vc = bits(c["k_cache"]).copy(), bits(c["v_cache"]).copy()
    assert oracle.append(kc, vc, bits(c["k_new"]), bits(c["v_new"]), slots) == -2


# ---------------------------------------------------------------- multi-query (causal)

def _causal_brute_force(q, k, v, n, scale):
    """Contiguous causal attention for one sequence and one head, pure Python loops:
    query token i of a chunk of L new tokens sees positions 0 .. n - L + i."""
    L = q.shape[0]
    out = np.zeros_like(q)
    for i in range(L):
        last = n - L + i
        scores = [scale * float(np.dot(q[i], k[t])) for t in range(last + 1)]
        m = max(scores)
        w = [math.exp(x - m) for x in scores]
        z = sum(w)
        for t in range(last + 1):
            out[i] += w[t] / z * v[t]
    return out


def test_multi_query_equals_causal_brute_force():
    w = make_workload("c1")
    s = w.spec
    q_len = 4
    q = make_queries(w, q_len, seed=3)
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    bt = w.block_tables.numpy()
    cl = w.context_lens.numpy()
    got = oracle.multi_query_attention(bits(q), kc, vc, bt, cl, w.scale, s.dtype)
    qv = oracle.decode_values(bits(q), s.dtype)
    group = s.num_q_heads // s.num_kv_heads
    for b in range(s.num_seqs):
        n = int(cl[b])
        for h in range(s.num_q_heads):
            k, v = oracle.gather_kv(kc, vc, bt, n, b, h // group)
            kd = oracle.decode_values(k, s.dtype)
            vd = oracle.decode_values(v, s.dtype)
            ref = _causal_brute_force(qv[b, :, h], kd, vd, n, w.scale)
            assert np.allclose(got[b, :, h], ref, rtol=1e-12, atol=1e-13)


def test_multi_query_of_one_token_is_decode_attention():
    w = make_workload("c1")
    q = make_queries(w, 1, seed=5)
    args = (bits(w.k_cache), bits(w.v_cache), w.block_tables.numpy(), w.context_lens.numpy(),
            w.scale, w.spec.dtype)
    mq = oracle.multi_query_attention(bits(q), *args)
    dec = oracle.decode_attention(bits(q)[:, 0], *args)
    assert np.array_equal(mq[:, 0], dec)


def test_multi_query_last_token_sees_whole_context_first_sees_less():
    w = make_workload("c1")
    q_len = 3
    q = make_queries(w, q_len, seed=7)
    kc, vc, bt, cl = bits(w.k_cache), bits(w.v_cache), w.block_tables.numpy(), w.context_lens.numpy()
    mq = oracle.multi_query_attention(bits(q), kc, vc, bt, cl, w.scale, w.spec.dtype)
    full = oracle.decode_attention(bits(q)[:, -1], kc, vc, bt, cl, w.scale, w.spec.dtype)
    first = oracle.decode_attention(bits(q)[:, 0], kc, vc, bt, cl - (q_len - 1), w.scale,
                                    w.spec.dtype)
    assert np.array_equal(mq[:, -1], full)
    assert np.array_equal(mq[:, 0], first)


# ---------------------------------------------------------------- FP8 (E4M3) cache

def test_e4m3_decoder_matches_library_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2   # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], lib[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encoder_round_trips_and_matches_library_rounding():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    values = oracle.decode_e4m3(codes).astype(np.float32)
    back = oracle.encode_e4m3(values)
    # every finite code comes back (0x80, negative zero, stays negative zero)
    assert np.array_equal(back, codes)
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(200000, generator=g) * torch.exp2(torch.randint(-12, 9, (200000,),
                                                                       generator=g).float()))
    x = x.clamp(-448, 448)
    ours = oracle.encode_e4m3(x.numpy())
    lib = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)


def test_e4m3_encoder_ties_saturation_and_nan():
    f = np.float32
    cases = {
        1.0625: 0x38,        # halfway 1.0 (0x38) / 1.125 (0x39): to the even code
        1.1875: 0x3A,        # halfway 1.125 / 1.25: to 1.25 (0x3A, even)
        2.0 ** -10: 0x00,    # halfway 0 / 2^-9: to zero (even)
        3 * 2.0 ** -10: 0x02,  # halfway 2^-9 / 2^-8: to 2^-8 (code 2, even)
        464.0: 0x7E,         # halfway 448 / (480, not a value): saturates
        1.0e6: 0x7E, -1.0e6: 0xFE,
        float("inf"): 0x7E, float("-inf"): 0xFE,
    }
    x = np.array(list(cases), dtype=f)
    assert list(oracle.encode_e4m3(x)) == list(cases.values())
    assert oracle.encode_e4m3(np.array([np.nan], dtype=f))[0] == 0x7F


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_append_fp8_matches_independent_quantisation(dtype):
    c = make_append_case(50, 8, 16, 4, 64, dtype, seed=9)
    k_new, v_new = c["k_new"], c["v_new"]
    slots = c["slot_mapping"].numpy()
    k_scale, v_scale = 0.0123, 0.0311
    kc = np.full((8, 16, 4, 64), 0x5A, dtype=np.uint8)
    vc = kc.copy()
    assert oracle.append_fp8(kc, vc, bits(k_new), bits(v_new), slots, k_scale, v_scale,
                             dtype) == 0
    ks = torch.full((8 * 16, 4, 64), 0x5A, dtype=torch.uint8)
    vs = ks.clone()
    for i, s in enumerate(slots):
        if s < 0:
            continue
        ks[s] = (k_new[i].float() / torch.tensor(k_scale, dtype=torch.float32)).clamp(
            -448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        vs[s] = (v_new[i].float() / torch.tensor(v_scale, dtype=torch.float32)).clamp(
            -448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(kc.reshape(8 * 16, 4, 64), ks.numpy())
    assert np.array_equal(vc.reshape(8 * 16, 4, 64), vs.numpy())


def test_decode_attention_fp8_equals_dense_attention_on_dequantized_values():
    w = make_workload("c3", num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=64,
                      lengths=("uniform", 5, 90), max_len_cap=96, seed=17)
    k_scale, v_scale = 5.0 / 448, 4.0 / 448
    kc = oracle.encode_e4m3(w.k_cache.float().numpy() / np.float32(k_scale))
    vc = oracle.encode_e4m3(w.v_cache.float().numpy() / np.float32(v_scale))
    bt, cl = w.block_tables.numpy(), w.context_lens.numpy()
    got = oracle.decode_attention_fp8(bits(w.q), kc, vc, bt, cl, w.scale, k_scale, v_scale,
                                      w.spec.dtype)
    kd = oracle.decode_e4m3(kc) * k_scale
    vd = oracle.decode_e4m3(vc) * v_scale
    qd = oracle.decode_values(bits(w.q), w.spec.dtype)
    group = w.spec.num_q_heads // w.spec.num_kv_heads
    for b in range(w.spec.num_seqs):
        n = int(cl[b])
        for h in range(w.spec.num_q_heads):
            k, v = oracle.gather_kv(kd, vd, bt, n, b, h // group)
            s = torch.from_numpy(qd[b, h] @ k.T * w.scale)
            ref = (torch.softmax(s, dim=0) @ torch.from_numpy(v)).numpy()
            assert np.allclose(got[b, h], ref, rtol=1e-12, atol=1e-14)
