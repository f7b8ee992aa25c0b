"""One-launch append + decode, and decode steps captured in CUDA graphs.

The fused call must leave the cache exactly as pkv_append through the
workload's slot_mapping would (bit for bit) and produce the decode result the
oracle computes after that append.  A captured step must replay to the same
bits as the same calls made eagerly on an identical workload.
"""
import pytest
import torch

import paged_kv_cache_164_gb300 as pkv
from helpers import assert_attention_close, oracle_after_append
from workloads import make_workload

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_fp16_d64": dict(name="c1"),
    "gqa8_bf16_split": dict(name="c3", num_seqs=6, lengths=("uniform", 100, 1500),
                            max_len_cap=1536, seed=71),
    "mha_fp16_d128": dict(name="c2", num_seqs=5, num_q_heads=8, num_kv_heads=8,
                          lengths=("uniform", 16, 700), max_len_cap=768, seed=72),
    "bs32_gqa4": dict(name="c5_bs32", num_seqs=7, lengths=("uniform", 31, 900), max_len_cap=960,
                      shared_prefix_groups=0, seed=73),
}


def _make(key, **kw):
    case = dict(CASES[key])
    name = case.pop("name")
    case.update(kw)
    return make_workload(name, device="cuda", **case)


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("key", sorted(CASES))
def test_fused_append_decode_matches_oracle_and_separate_append(key, splits):
    w = _make(key, poison=True)
    expect, _, _ = oracle_after_append(w)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    pkv.append(w.k_new, w.v_new, kc, vc, w.slot_mapping)
    flag = pkv.new_error_flag("cuda")
    out = pkv.append_decode_attention(w.q, w.k_new, w.v_new, w.k_cache, w.v_cache,
                                      w.block_tables, w.context_lens, w.max_context_len,
                                      scale=w.scale, num_splits=splits, err_flag=flag)
    assert pkv.check_error(flag) == 0
    # the cache holds exactly what the separate append writes (NaN bit patterns included)
    assert torch.equal(w.k_cache.view(torch.int16), kc.view(torch.int16))
    assert torch.equal(w.v_cache.view(torch.int16), vc.view(torch.int16))
    assert_attention_close(out, expect, f"{key} splits={splits}")


def test_fused_append_skips_and_flags_a_bad_last_block():
    w = _make("gqa8_bf16_split")
    before = w.k_cache.clone()
    bt = w.block_tables.clone()
    b = 2
    n = int(w.context_lens[b])
    bt[b, (n - 1) // w.spec.block_size] = w.num_blocks + 5   # out of range
    flag = pkv.new_error_flag("cuda")
    pkv.append_decode_attention(w.q, w.k_new, w.v_new, w.k_cache, w.v_cache, bt, w.context_lens,
                                w.max_context_len, scale=w.scale, err_flag=flag)
    assert pkv.check_error(flag) & pkv.EFLAG_BLOCK_ID
    # only the other sequences' new slots changed
    changed = (w.k_cache.view(torch.int16) != before.view(torch.int16)).any(dim=(2, 3))
    slots = w.slot_mapping.cpu().tolist()
    bs = w.spec.block_size
    expect_changed = {(s // bs, s % bs) for i, s in enumerate(slots) if i != b}
    got_changed = {tuple(x) for x in torch.nonzero(changed).cpu().tolist()}
    assert got_changed <= expect_changed


def _graph_vs_eager(make, step, steps=3):
    """Runs ``step`` eagerly on one workload and from a captured graph on its twin."""
    wa, wb = make(), make()
    outs_a = []
    for i in range(steps):
        torch.manual_seed(100 + i)
        wa.q.copy_(torch.randn_like(wa.q, dtype=torch.float32).to(wa.q.dtype))
        outs_a.append(step(wa).clone())
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(wb)                       # first calls (library set-up) outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    # restore wb's cache to the untouched twin so both start from the same state
    fresh = make()
    wb.k_cache.copy_(fresh.k_cache)
    wb.v_cache.copy_(fresh.v_cache)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out_b = step(wb)
    for i in range(steps):
        torch.manual_seed(100 + i)
        wb.q.copy_(torch.randn_like(wb.q, dtype=torch.float32).to(wb.q.dtype))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_b, outs_a[i]), f"replay {i} differs from the eager step"
    assert torch.equal(wb.k_cache.view(torch.int16), wa.k_cache.view(torch.int16))


def test_graph_of_fused_step_replays_like_eager():
    def make():
        w = _make("gqa8_bf16_split")
        s = w.spec
        w._ws = torch.empty(max(16, pkv.workspace_size(s.num_seqs, s.num_q_heads, s.num_kv_heads,
                                                       s.head_dim, s.block_size,
                                                       w.max_context_len, 0)),
                            dtype=torch.uint8, device="cuda")
        w._out = torch.empty_like(w.q)
        w._mcl = w.max_context_len
        return w

    def step(w):
        return pkv.append_decode_attention(w.q, w.k_new, w.v_new, w.k_cache, w.v_cache,
                                           w.block_tables, w.context_lens, w._mcl,
                                           scale=w.scale, out=w._out, workspace=w._ws)
    _graph_vs_eager(make, step)


def test_graph_of_append_then_decode_replays_like_eager():
    def make():
        w = _make("mha_fp16_d128")
        s = w.spec
        w._ws = torch.empty(max(16, pkv.workspace_size(s.num_seqs, s.num_q_heads, s.num_kv_heads,
                                                       s.head_dim, s.block_size,
                                                       w.max_context_len, 0)),
                            dtype=torch.uint8, device="cuda")
        w._out = torch.empty_like(w.q)
        w._mcl = w.max_context_len
        return w

    def step(w):
        pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
        return pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                    w._mcl, scale=w.scale, out=w._out, workspace=w._ws)
    _graph_vs_eager(make, step)


def test_graph_of_shared_prefix_step_replays_like_eager():
    def make():
        w = make_workload("c5", device="cuda", num_seqs=16,
                          lengths=("prefix_lognormal", 256, 300, 1.0, 1500), max_len_cap=1536,
                          shared_prefix_groups=2)
        s = w.spec
        w._mgs, w._mpl, w._mcl = w.max_group_size, w.max_prefix_len, w.max_context_len
        w._ws = torch.empty(pkv.prefix_shared_workspace_size(
            s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim, s.block_size, w._mcl,
            w.group_prefix_len.numel(), w._mgs, w._mpl), dtype=torch.uint8, device="cuda")
        w._out = torch.empty_like(w.q)
        return w

    def step(w):
        pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
        return pkv.decode_attention_prefix_shared(
            w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w._mcl, w.group_start,
            w.group_prefix_len, w._mgs, w._mpl, scale=w.scale, out=w._out, workspace=w._ws)
    _graph_vs_eager(make, step)


@pytest.mark.parametrize("q_len", [2, 8])   # 16 rows: decode kernel; 64 rows: tcgen05 kernel
def test_graph_of_multi_query_step_replays_like_eager(q_len):
    from workloads import make_queries

    def make():
        w = make_workload("c3", device="cuda", num_seqs=3, lengths=("uniform", 300, 1400),
                          max_len_cap=1536, seed=74)
        s = w.spec
        w.q = make_queries(w, q_len, seed=75)
        w._mcl = w.max_context_len
        w._ws = torch.empty(max(16, pkv.multi_query_workspace_size(
            s.num_seqs, q_len, s.num_q_heads, s.num_kv_heads, s.head_dim, s.block_size,
            w._mcl)), dtype=torch.uint8, device="cuda")
        w._out = torch.empty_like(w.q)
        return w

    def step(w):
        return pkv.multi_query_attention(w.q, w.k_cache, w.v_cache, w.block_tables,
                                         w.context_lens, w._mcl, scale=w.scale, out=w._out,
                                         workspace=w._ws)
    _graph_vs_eager(make, step)


def test_graph_of_e4m3_append_then_decode_replays_like_eager():
    import numpy as np

    import oracle
    k_scale, v_scale = 5.0 / 448, 4.5 / 448

    def make():
        w = make_workload("c3", device="cuda", num_seqs=4, lengths=("uniform", 100, 900),
                          max_len_cap=960, seed=76)
        s = w.spec
        w.k_cache = torch.from_numpy(oracle.encode_e4m3(
            w.k_cache.float().cpu().numpy() / np.float32(k_scale))).cuda()
        w.v_cache = torch.from_numpy(oracle.encode_e4m3(
            w.v_cache.float().cpu().numpy() / np.float32(v_scale))).cuda()
        w._mcl = w.max_context_len
        w._ws = torch.empty(max(16, pkv.workspace_size(s.num_seqs, s.num_q_heads,
                                                       s.num_kv_heads, s.head_dim, s.block_size,
                                                       w._mcl, 0)),
                            dtype=torch.uint8, device="cuda")
        w._out = torch.empty_like(w.q)
        return w

    def step(w):
        pkv.append_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, k_scale, v_scale)
        return pkv.decode_attention_fp8(w.q, w.k_cache, w.v_cache, w.block_tables,
                                        w.context_lens, w._mcl, k_scale, v_scale, scale=w.scale,
                                        out=w._out, workspace=w._ws)
    _graph_vs_eager(make, step)


def test_graph_of_fused_e4m3_step_replays_like_eager():
    import numpy as np

    import oracle
    k_scale, v_scale = 5.0 / 448, 4.5 / 448

    def make():
        w = make_workload("c3", device="cuda", num_seqs=4, lengths=("uniform", 100, 900),
                          max_len_cap=960, seed=77)
        s = w.spec
        w.k_cache = torch.from_numpy(oracle.encode_e4m3(
            w.k_cache.float().cpu().numpy() / np.float32(k_scale))).cuda()
        w.v_cache = torch.from_numpy(oracle.encode_e4m3(
            w.v_cache.float().cpu().numpy() / np.float32(v_scale))).cuda()
        w._mcl = w.max_context_len
        w._ws = torch.empty(max(16, pkv.workspace_size(s.num_seqs, s.num_q_heads,
                                                       s.num_kv_heads, s.head_dim, s.block_size,
                                                       w._mcl, 0)),
                            dtype=torch.uint8, device="cuda")
        w._out = torch.empty_like(w.q)
        return w

    def step(w):
        return pkv.append_decode_attention_fp8(w.q, w.k_new, w.v_new, w.k_cache, w.v_cache,
                                               w.block_tables, w.context_lens, w._mcl, k_scale,
                                               v_scale, scale=w.scale, out=w._out,
                                               workspace=w._ws)
    _graph_vs_eager(make, step)
