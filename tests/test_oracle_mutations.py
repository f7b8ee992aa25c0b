"""Plants mistakes in copies of the C oracle (on the CPU) and checks the pins catch them.

Each mutant is the oracle's source with one plausible slip — a dropped scale, a
wrong GQA head index, block and offset swapped, V read from the K cache, no
max subtraction, a dropped token, a missing normalisation, a wrong fp16
exponent bias or a wrong bf16 shift — compiled into a temporary directory.
The same independent references the pin tests use (library conversion, dense
torch attention, the dominant-key closed form) must reject every mutant, while
the unmodified source passes them.  The E4M3 functions get their own mutants
(exponent bias, subnormal scale, ties away from even, saturation losing its
sign, the append's scales, the attention's scales), rejected by references that
do not use them: torch's float8_e4m3fn type, tie and saturation codes worked out
from the format, an independent quantising scatter, and dense torch attention
over values the torch type dequantises.  The multi-query (causal) function,
plain Python over the decode oracle, is mutated in copies of its source (a
limit one short, the causal order reversed, rows paired with the wrong
sequences' tables) and must fail the causal brute force.  The pages' combine
and the log-sum-exp merge (plain Python too) are mutated the same way (the
segment scales dropped from L*, unweighted partials, empty splits weighted,
base-2 weights of natural-log lse, no final division) and must fail the
split / merge pins.  The append scatter (C) and the block-table gather (Python)
get mutants too (V rows from the new K rows, the in-block offset dropped, block
and offset exchanged; the page index shifted by a token, V read from the K
cache, always the first KV head), rejected by the independent scatter and by
the pages' block-table example plus dense attention over gathered rows.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import build as oracle_build
from oracle.reference import load_library
from workloads import bits, make_append_case, make_queries, make_workload

from test_oracle_pins import SMALL_CASES, _dense_torch, _make

MUTANTS = {
    "drop_scale": ("s[t] = scale * dot;", "s[t] = dot;"),
    "gqa_modulo": ("const int g = h / group;", "const int g = h % num_kv_heads;"),
    "block_offset_swapped": ("int off = t % block_size;\n                if (blk",
                             "int off = t / block_size % block_size;\n                if (blk"),
    "v_from_k_cache": ("v_cache + (((int64_t)blk", "k_cache + (((int64_t)blk"),
    "no_max_subtraction": ("s[t] = exp(s[t] - m);", "s[t] = exp(s[t]);"),
    "drop_last_token": ("const int n = context_lens[b];", "const int n = context_lens[b] - 1;"),
    "no_normalisation": ("double w = s[t] / z;", "double w = s[t];"),
    "fp16_bias": ("expo - 25", "expo - 24"),
    "bf16_shift": ("((uint32_t)b) << 16", "((uint32_t)b) << 15"),
}


def _compile(tmp_path, name, src):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(c), "-lm"], check=True)
    return load_library(str(so))


def _fails_a_pin(lib) -> bool:
    """True if the library disagrees with one of the independent references."""
    raw = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dtype, tdt in (("fp16", torch.float16), ("bf16", torch.bfloat16)):
        ref = torch.from_numpy(raw.view(np.int16).copy()).view(tdt).to(torch.float64).numpy()
        got = oracle.decode_values(raw, dtype, lib=lib)
        fin = np.isfinite(ref)
        if not np.array_equal(got[fin], ref[fin]):
            return True
    for case in SMALL_CASES:
        w = _make(case)
        try:
            got = oracle.decode_attention(bits(w.q), bits(w.k_cache), bits(w.v_cache),
                                          w.block_tables.numpy(), w.context_lens.numpy(),
                                          w.scale, w.spec.dtype, lib=lib)
        except ValueError:
            return True
        if not np.allclose(got, _dense_torch(w), rtol=0, atol=1e-9):
            return True
    # dominant key with a huge score gap (closed form: the output is that key's value)
    w = make_workload("c3", num_seqs=1, num_q_heads=2, num_kv_heads=1, head_dim=64,
                      lengths=("fixed", (40,)), max_len_cap=40, pool="free_list",
                      pool_slack=1.0, seed=7)
    k_cache = w.k_cache.clone()
    q = torch.zeros_like(w.q)
    q[0, :, 0] = 64.0
    k_cache[:, :, :, 0] = 1.0
    blk = int(w.block_tables[0, 1])
    k_cache[blk, 13, 0, 0] = 256.0
    got = oracle.decode_attention(bits(q), bits(k_cache), bits(w.v_cache),
                                  w.block_tables.numpy(), w.context_lens.numpy(), w.scale,
                                  w.spec.dtype, lib=lib)
    v_star = w.v_cache[blk, 13, 0].to(torch.float64).numpy()
    return not np.array_equal(got[0, 0], v_star)


@pytest.fixture(scope="module")
def source():
    with open(oracle_build.SRC) as f:
        return f.read()


def test_unmodified_source_passes(tmp_path, source):
    assert not _fails_a_pin(_compile(tmp_path, "original", source))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, source, name):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation site for {name} not found"
    mutated = source.replace(old, new, 1)
    assert mutated != source
    assert _fails_a_pin(_compile(tmp_path, name, mutated)), f"pins miss mutant {name}"


# ---------------------------------------------------------------- E4M3 (FP8) functions

E4M3_MUTANTS = {
    "e4m3_exponent_bias": ("ldexp((double)(8 + frac), expo - 10)",
                           "ldexp((double)(8 + frac), expo - 11)"),
    "e4m3_subnormal_scale": ("ldexp((double)frac, -9)", "ldexp((double)frac, -10)"),
    "e4m3_ties_away_from_even": ("return fmod(f, 2.0) == 0.0 ? f : f + 1.0;", "return f + 1.0;"),
    "e4m3_saturation_drops_sign": ("if (a >= 448.0) return sign | 0x7E;",
                                   "if (a >= 448.0) return 0x7E;"),
    "fp8_append_unscaled": ("k_cache[dst + j] = encode_e4m3(kx / k_scale);",
                            "k_cache[dst + j] = encode_e4m3(kx);"),
    "fp8_append_v_with_k_scale": ("v_cache[dst + j] = encode_e4m3(vx / v_scale);",
                                  "v_cache[dst + j] = encode_e4m3(vx / k_scale);"),
    "fp8_attention_k_unscaled": ("dot += qd[j] * (decode_e4m3(kt[j]) * k_scale);",
                                 "dot += qd[j] * decode_e4m3(kt[j]);"),
    "fp8_attention_v_unscaled": ("o[j] += w * (decode_e4m3(vt[j]) * v_scale);",
                                 "o[j] += w * decode_e4m3(vt[j]);"),
}


def _lib_e4m3(x: torch.Tensor) -> torch.Tensor:
    """The library's E4M3 codes of x (round to nearest even; x within +-448)."""
    return x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)


def _fails_an_e4m3_pin(lib) -> bool:
    """True if the library's E4M3 functions disagree with a reference that does
    not use them: torch's float8_e4m3fn type, the tie / saturation codes worked
    out from the format, an independent quantising scatter, and dense torch
    attention over values the torch type dequantises."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(codes, lib=lib)
    fin = np.isfinite(ref)
    if not np.array_equal(got[fin], ref[fin]) or not np.isnan(got[~fin]).all():
        return True
    g = torch.Generator().manual_seed(6)
    x = torch.randn(50000, generator=g) * torch.exp2(
        torch.randint(-12, 9, (50000,), generator=g).float())
    x = x.clamp(-448, 448)
    if not np.array_equal(oracle.encode_e4m3(x.numpy(), lib=lib), _lib_e4m3(x).numpy()):
        return True
    # ties to the even code, the subnormal tie, saturation with its sign
    worked = {1.0625: 0x38, 1.1875: 0x3A, 3 * 2.0 ** -10: 0x02, 470.0: 0x7E, -1.0e6: 0xFE}
    enc = oracle.encode_e4m3(np.array(list(worked), dtype=np.float32), lib=lib)
    if list(enc) != list(worked.values()):
        return True
    # quantising append against an independent scatter
    c = make_append_case(40, 8, 16, 2, 32, "bf16", seed=11)
    slots = c["slot_mapping"].numpy()
    k_scale, v_scale = 0.0123, 0.0311
    kc = np.full((8, 16, 2, 32), 0x5A, dtype=np.uint8)
    vc = kc.copy()
    if oracle.append_fp8(kc, vc, bits(c["k_new"]), bits(c["v_new"]), slots, k_scale, v_scale,
                         "bf16", lib=lib) != 0:
        return True
    ks = torch.full((8 * 16, 2, 32), 0x5A, dtype=torch.uint8)
    vs = ks.clone()
    for i, s in enumerate(slots):
        if s >= 0:
            ks[s] = _lib_e4m3(c["k_new"][i].float() / torch.tensor(k_scale))
            vs[s] = _lib_e4m3(c["v_new"][i].float() / torch.tensor(v_scale))
    if not (np.array_equal(kc.reshape(-1, 2, 32), ks.numpy()) and
            np.array_equal(vc.reshape(-1, 2, 32), vs.numpy())):
        return True
    # attention over an E4M3 cache against dense torch attention
    w = make_workload("c3", num_seqs=2, num_q_heads=4, num_kv_heads=2, head_dim=32,
                      lengths=("uniform", 5, 60), max_len_cap=64, seed=19)
    k_scale, v_scale = 5.0 / 448, 4.0 / 448
    kq = _lib_e4m3(w.k_cache.float() / k_scale)
    vq = _lib_e4m3(w.v_cache.float() / v_scale)
    bt, cl = w.block_tables.numpy(), w.context_lens.numpy()
    got = oracle.decode_attention_fp8(bits(w.q), kq.numpy(), vq.numpy(), bt, cl, w.scale,
                                      k_scale, v_scale, w.spec.dtype, lib=lib)
    kd = kq.view(torch.float8_e4m3fn).to(torch.float64) * k_scale
    vd = vq.view(torch.float8_e4m3fn).to(torch.float64) * v_scale
    qd = w.q.to(torch.float64)
    bs = w.spec.block_size
    for b in range(2):
        n = int(cl[b])
        t = torch.arange(n)
        blk = torch.from_numpy(bt[b]).long()[t // bs]
        for h in range(4):
            k = kd[blk, t % bs, h // 2]
            v = vd[blk, t % bs, h // 2]
            ref = torch.softmax(qd[b, h] @ k.T * w.scale, dim=0) @ v
            if not np.allclose(got[b, h], ref.numpy(), rtol=1e-12, atol=1e-14):
                return True
    return False


def test_unmodified_source_passes_the_e4m3_pins(tmp_path, source):
    assert not _fails_an_e4m3_pin(_compile(tmp_path, "original_e4m3", source))


@pytest.mark.parametrize("name", sorted(E4M3_MUTANTS))
def test_e4m3_mutant_is_caught(tmp_path, source, name):
    old, new = E4M3_MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not found once"
    mutated = source.replace(old, new)
    assert _fails_an_e4m3_pin(_compile(tmp_path, name, mutated)), f"pins miss mutant {name}"


# ---------------------------------------------------------------- multi-query (causal) attention

MQ_MUTANTS = {
    "mq_limit_one_short": ("cl[:, None] - q_len + 1 + np.arange(q_len)",
                           "cl[:, None] - q_len + np.arange(q_len)"),
    "mq_causal_order_reversed": ("np.arange(q_len)[None, :]", "np.arange(q_len)[::-1][None, :]"),
    "mq_tables_tiled": ("np.repeat(np.asarray(block_tables), q_len, axis=0)",
                        "np.tile(np.asarray(block_tables), (q_len, 1))"),
}


def _mq_function(src: str):
    """The oracle's multi_query_attention compiled from `src`, in its module's namespace."""
    import oracle.reference as ref
    ns = dict(ref.__dict__)
    exec(compile(src, "mutant", "exec"), ns)
    return ns["multi_query_attention"]


def _fails_the_causal_pin(mq) -> bool:
    """True if `mq` disagrees with the causal brute force of the pin tests on two
    sequences with their own tables and four query tokens."""
    from test_oracle_pins import _causal_brute_force
    w = make_workload("c1")
    s = w.spec
    q_len = 4
    q = make_queries(w, q_len, seed=3)
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    bt, cl = w.block_tables.numpy(), w.context_lens.numpy()
    try:
        got = mq(bits(q), kc, vc, bt, cl, w.scale, s.dtype)
    except ValueError:
        return True
    qv = oracle.decode_values(bits(q), s.dtype)
    group = s.num_q_heads // s.num_kv_heads
    for b in range(s.num_seqs):
        n = int(cl[b])
        for h in range(s.num_q_heads):
            k, v = oracle.gather_kv(kc, vc, bt, n, b, h // group)
            ref = _causal_brute_force(qv[b, :, h], oracle.decode_values(k, s.dtype),
                                      oracle.decode_values(v, s.dtype), n, w.scale)
            if not np.allclose(got[b, :, h], ref, rtol=1e-12, atol=1e-13):
                return True
    return False


def test_unmodified_multi_query_passes_the_causal_pin():
    import inspect
    import oracle.reference as ref
    assert not _fails_the_causal_pin(_mq_function(inspect.getsource(ref.multi_query_attention)))


@pytest.mark.parametrize("name", sorted(MQ_MUTANTS))
def test_multi_query_mutant_is_caught(name):
    import inspect
    import oracle.reference as ref
    src = inspect.getsource(ref.multi_query_attention)
    old, new = MQ_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found once"
    assert _fails_the_causal_pin(_mq_function(src.replace(old, new))), f"pin misses {name}"


# ---------------------------------------------------------------- combine and log-sum-exp merge

MERGE_MUTANTS = {
    "combine_drops_segment_scales_in_sum": ("l_star = np.sum(scale_i * l_sum)",
                                            "l_star = np.sum(l_sum)"),
    "combine_unweighted_partials": ("(scale_i * (l_sum / l_star))[:, None] * o",
                                    "(l_sum / l_star)[:, None] * o"),
    "merge_empty_split_weighted": (
        "w = np.where(np.isfinite(pl), np.exp(np.where(np.isfinite(pl), pl, 0.0) - safe_star), 0.0)",
        "w = np.exp(np.where(np.isfinite(pl), pl, 0.0) - safe_star)"),
    "merge_base_two_weights": ("np.exp(np.where(np.isfinite(pl), pl, 0.0) - safe_star)",
                               "np.exp2(np.where(np.isfinite(pl), pl, 0.0) - safe_star)"),
    "merge_unnormalised": ("num / np.where(den > 0, den, 1.0)", "num"),
}


def _merge_source() -> str:
    import inspect
    import oracle.reference as ref
    return "\n\n".join(inspect.getsource(f) for f in (ref.combine_result, ref.merge_lse,
                                                        ref.decode_attention_pagewise))


def _merge_functions(src: str):
    """combine_result, merge_lse and decode_attention_pagewise compiled from `src`
    in a copy of their module's namespace (so the pagewise decode calls the
    combine compiled here)."""
    import oracle.reference as ref
    ns = dict(ref.__dict__)
    exec(compile(src, "mutant", "exec"), ns)
    return ns["combine_result"], ns["merge_lse"], ns["decode_attention_pagewise"]


def _fails_a_merge_pin(combine, merge, pagewise) -> bool:
    """True if the functions disagree with the pins of the split / merge tests:
    the pages' per-page decode and random splits equal the single pass, and the
    merge's worked edge cases."""
    from test_oracle_pins import SMALL_CASES, _make, _np, _oracle
    for case in SMALL_CASES:
        w = _make(case)
        got = pagewise(_np(w.q), _np(w.k_cache), _np(w.v_cache), w.block_tables.numpy(),
                       w.context_lens.numpy(), w.scale)
        if not np.allclose(got, _oracle(w), rtol=0, atol=1e-13):
            return True
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
            if not np.allclose(combine(o, l_sum, m), full[b, h], rtol=0, atol=1e-13):
                return True
            lse = np.where(np.isfinite(m), m + np.log(np.where(l_sum > 0, l_sum, 1.0)), -np.inf)
            if not np.allclose(merge(o, lse), full[b, h], rtol=0, atol=1e-13):
                return True
    o = np.array([[1.0, 2.0], [3.0, 4.0]])
    edge = [([-np.inf, -np.inf], [0.0, 0.0]), ([-np.inf, 0.3], [3.0, 4.0]),
            ([0.0, 0.0], [2.0, 3.0]), ([math.log(3.0), 0.0], [1.5, 2.5])]
    return any(not np.allclose(merge(o, np.array(lse)), out, rtol=1e-15, atol=0)
               for lse, out in edge)


def test_unmodified_merge_functions_pass_the_merge_pins():
    assert not _fails_a_merge_pin(*_merge_functions(_merge_source()))


@pytest.mark.parametrize("name", sorted(MERGE_MUTANTS))
def test_merge_mutant_is_caught(name):
    src = _merge_source()
    old, new = MERGE_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found once"
    assert _fails_a_merge_pin(*_merge_functions(src.replace(old, new))), f"pins miss {name}"


# ---------------------------------------------------------------- append scatter and gather

APPEND_MUTANTS = {
    "append_v_from_k_new": ("memcpy(v_cache + dst, v_new + (int64_t)i * row",
                            "memcpy(v_cache + dst, k_new + (int64_t)i * row"),
    "append_offset_dropped": ("int64_t dst = (blk * block_size + off) * row;",
                              "int64_t dst = (blk * block_size) * row;"),
    "append_block_as_offset": ("int64_t dst = (blk * block_size + off) * row;",
                               "int64_t dst = (off * block_size + blk % block_size) * row;"),
}

GATHER_MUTANTS = {
    "gather_page_shifted": ("blk = block_tables[seq, t // bs]",
                            "blk = block_tables[seq, (t + 1) // bs]"),
    "gather_v_from_k_cache": ("v_cache[blk, off, kv_head, :]", "k_cache[blk, off, kv_head, :]"),
    "gather_first_kv_head": ("k_cache[blk, off, kv_head, :]", "k_cache[blk, off, 0, :]"),
}


def _fails_the_append_pin(lib) -> bool:
    """The append pin: an independent numpy scatter, and untouched slots keep the
    sentinel (every mutant keeps its writes inside the pool)."""
    for dtype in ("fp16", "bf16"):
        c = make_append_case(300, 40, 16, 4, 64, dtype, seed=5)
        kc, vc = bits(c["k_cache"]).copy(), bits(c["v_cache"]).copy()
        slots = c["slot_mapping"].numpy()
        if oracle.append(kc, vc, bits(c["k_new"]), bits(c["v_new"]), slots, lib=lib) != 0:
            return True
        ek, ev = bits(c["k_cache"]).copy(), bits(c["v_cache"]).copy()
        keep = slots >= 0
        ek.reshape(-1, 4, 64)[slots[keep]] = bits(c["k_new"])[keep]
        ev.reshape(-1, 4, 64)[slots[keep]] = bits(c["v_new"])[keep]
        if not (np.array_equal(kc, ek) and np.array_equal(vc, ev)):
            return True
    return False


def test_unmodified_append_passes_its_pin(tmp_path, source):
    assert not _fails_the_append_pin(_compile(tmp_path, "original_append", source))


@pytest.mark.parametrize("name", sorted(APPEND_MUTANTS))
def test_append_mutant_is_caught(tmp_path, source, name):
    old, new = APPEND_MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not found once"
    lib = _compile(tmp_path, name, source.replace(old, new))
    assert _fails_the_append_pin(lib), f"pin misses mutant {name}"


def _gather_function(src: str):
    import oracle.reference as ref
    ns = dict(ref.__dict__)
    exec(compile(src, "mutant", "exec"), ns)
    return ns["gather_kv"]


def _fails_a_gather_pin(gather) -> bool:
    """The gather pins: the pages' block-table worked example (golden file), and
    on a two-KV-head workload with its own K and V, the rows the decode
    definition reads (the oracle's dense attention over gathered rows equals its
    paged attention)."""
    from test_oracle_pins import GOLDEN, _make, _np, _oracle
    table, bs = {}, None
    with open(os.path.join(GOLDEN, "block_table_example.txt")) as f:
        for line in f:
            p = line.split()
            if not p or p[0].startswith("#"):
                continue
            if p[0] == "block_size":
                bs = int(p[1])
                continue
            table.setdefault(int(p[0]), {})[int(p[1])] = int(p[2])
    cache = np.zeros((8, bs, 1, 2), dtype=np.int32)
    cache[:, :, 0, 0] = np.arange(8)[:, None]
    cache[:, :, 0, 1] = np.arange(bs)[None, :]
    tables = np.full((2, 3), -1, dtype=np.int32)
    for req, m in table.items():
        for logical, phys in m.items():
            tables[req - 1, logical] = phys
    try:
        k, _ = gather(cache, cache, tables, 3 * bs, 0, 0)
    except IndexError:
        return True
    if k[:, 0].tolist() != [5] * bs + [7] * bs + [2] * bs or \
            k[:, 1].tolist() != list(range(bs)) * 3:
        return True
    w = _make(dict(name="c3", num_seqs=2, num_q_heads=4, num_kv_heads=2, head_dim=32,
                   lengths=("uniform", 20, 90), max_len_cap=96, pool="free_list", seed=23))
    paged = _oracle(w)
    q, kc, vc = _np(w.q), _np(w.k_cache), _np(w.v_cache)
    for b in range(2):
        n = int(w.context_lens[b])
        for h in range(4):
            try:
                k, v = gather(kc, vc, w.block_tables.numpy(), n, b, h // 2)
            except IndexError:
                return True
            s = torch.from_numpy(q[b, h] @ k.T * w.scale)
            dense = (torch.softmax(s, dim=0) @ torch.from_numpy(v)).numpy()
            if not np.allclose(dense, paged[b, h], rtol=1e-12, atol=1e-13):
                return True
    return False


def test_unmodified_gather_passes_its_pins():
    import inspect
    import oracle.reference as ref
    assert not _fails_a_gather_pin(_gather_function(inspect.getsource(ref.gather_kv)))


@pytest.mark.parametrize("name", sorted(GATHER_MUTANTS))
def test_gather_mutant_is_caught(name):
    import inspect
    import oracle.reference as ref
    src = inspect.getsource(ref.gather_kv)
    old, new = GATHER_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found once"
    assert _fails_a_gather_pin(_gather_function(src.replace(old, new))), f"pins miss {name}"
