"""Shared-prefix decode on the GPU against the fp64 oracle (the same definition).

Sequences come in contiguous groups whose first tokens are the same physical
blocks; the library reads each group's prefix once for all members.  The result
must be the plain decode-attention result, so the oracle is unchanged.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_164_gb300 as pkv
from helpers import assert_attention_close, oracle_after_append
from workloads import make_workload

pytestmark = pytest.mark.gpu


def _run(w, group_start=None, group_prefix_len=None, max_group_size=None, max_prefix_len=None,
         flag=None, append=True):
    if append:
        pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, err_flag=flag)
    gs = w.group_start if group_start is None else group_start
    gp = w.group_prefix_len if group_prefix_len is None else group_prefix_len
    return pkv.decode_attention_prefix_shared(
        w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.max_context_len, gs, gp,
        w.max_group_size if max_group_size is None else max_group_size,
        w.max_prefix_len if max_prefix_len is None else max_prefix_len, scale=w.scale,
        err_flag=flag)


CASES = {
    "bs16_g4_2groups": dict(name="c5", num_seqs=16, lengths=("prefix_lognormal", 256, 300, 1.0, 1500),
                            max_len_cap=1536, shared_prefix_groups=2),
    "bs32_g4_4groups": dict(name="c5_bs32", num_seqs=24, lengths=("prefix_lognormal", 512, 200, 1.0, 1200),
                            max_len_cap=1280, shared_prefix_groups=4),
    "mha_fp16_d128": dict(name="c2", num_seqs=12, num_q_heads=8, num_kv_heads=8,
                          lengths=("prefix_lognormal", 64, 100, 1.0, 600), max_len_cap=640,
                          shared_prefix_groups=3, seed=41),
    "gqa8_d64_bf16": dict(name="c3", num_seqs=8, num_q_heads=16, num_kv_heads=2, head_dim=64,
                          lengths=("prefix_lognormal", 128, 50, 1.0, 400), max_len_cap=512,
                          shared_prefix_groups=2, pool="free_list", seed=43),
    "gqa16_big_group": dict(name="c3", num_seqs=40, num_q_heads=32, num_kv_heads=2, head_dim=128,
                            lengths=("prefix_lognormal", 160, 40, 1.0, 300), max_len_cap=320,
                            shared_prefix_groups=1, pool="free_list", seed=47),
    # more than one plan-kernel chunk of groups and of (sequence, KV head) units
    "1100_groups_of_one": dict(name="c3", num_seqs=1100, num_q_heads=4, num_kv_heads=2, head_dim=64,
                               lengths=("prefix_lognormal", 16, 20, 0.5, 80), max_len_cap=96,
                               shared_prefix_groups=1100, pool="free_list", seed=53),
    # GQA group of 6: members' rows straddle the 128-row tiles of the prefix kernel
    # (member 21: rows 126-131), so such a unit gets contributions from two tiles
    "gqa6_rows_straddle_tiles": dict(name="c3", num_seqs=45, num_q_heads=12, num_kv_heads=2,
                                     head_dim=128, lengths=("prefix_lognormal", 160, 40, 1.0, 300),
                                     max_len_cap=320, shared_prefix_groups=1, seed=61),
    # more groups than the plan keeps in shared memory (4096): their bounds are read in place
    "4200_groups_of_one": dict(name="c3", num_seqs=4200, num_q_heads=2, num_kv_heads=1, head_dim=64,
                               lengths=("prefix_lognormal", 16, 10, 0.5, 48), max_len_cap=64,
                               shared_prefix_groups=4200, pool="free_list", seed=59),
}


def _make(key, **kw):
    case = dict(CASES[key])
    name = case.pop("name")
    case.update(kw)
    return make_workload(name, device="cuda", **case)


@pytest.mark.parametrize("key", sorted(CASES))
def test_shared_prefix_matches_oracle(key):
    w = _make(key, poison=True)
    expect, _, _ = oracle_after_append(w)
    flag = pkv.new_error_flag("cuda")
    out = _run(w, flag=flag)
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, expect, key)


def test_groups_of_one_and_no_prefix_equal_plain_decode():
    w = _make("bs16_g4_2groups")
    expect, _, _ = oracle_after_append(w)
    b = w.spec.num_seqs
    gs = torch.arange(0, b + 1, dtype=torch.int32, device="cuda")
    gp = torch.zeros(b, dtype=torch.int32, device="cuda")
    out = _run(w, gs, gp, 1, 0)
    assert_attention_close(out, expect, "groups of one")
    # mixed: the first group shared, the rest groups of one with no prefix
    half = b // 2
    gs2 = torch.tensor([0] + list(range(half, b + 1)), dtype=torch.int32, device="cuda")
    gp2 = torch.tensor([256] + [0] * (b - half), dtype=torch.int32, device="cuda")
    out2 = _run(w, gs2, gp2, half, 256, append=False)
    assert_attention_close(out2, expect, "mixed groups")


def test_member_shorter_than_the_prefix_is_masked():
    w = _make("bs16_g4_2groups")
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    cl = w.context_lens.clone()
    cl[3] = 100          # inside the 256-token prefix of group 0
    cl[9] = 256          # exactly the prefix of group 1
    w.context_lens = cl
    expect, _, _ = oracle_after_append(w)  # the oracle re-appends the same tokens: idempotent
    out = _run(w, append=False)
    assert_attention_close(out, expect, "short members")


def test_members_without_suffix_are_merged_by_the_prefix_kernel():
    # Every member of group 0 ends exactly at the shared prefix: no suffix
    # partition exists, so the prefix CTAs write each unit's last partial and
    # must merge it themselves.
    w = _make("bs32_g4_4groups")
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    cl = w.context_lens.clone()
    g0, g1 = int(w.group_start[0]), int(w.group_start[1])
    cl[g0:g1] = int(w.group_prefix_len[0])
    w.context_lens = cl
    expect, _, _ = oracle_after_append(w)
    flag = pkv.new_error_flag("cuda")
    out = _run(w, append=False, flag=flag)
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, expect, "no suffixes")


def test_malformed_group_is_flagged_and_still_correct():
    w = _make("bs32_g4_4groups")
    expect, _, _ = oracle_after_append(w)
    gp = w.group_prefix_len.clone()
    gp[1] = 17           # not a multiple of the block size
    flag = pkv.new_error_flag("cuda")
    out = _run(w, group_prefix_len=gp, flag=flag)
    assert pkv.check_error(flag) & pkv.EFLAG_GROUP
    assert_attention_close(out, expect, "malformed group falls back")


@pytest.mark.parametrize("name", ["c5", "c5_bs32"])
def test_full_size_shared_prefix_sampled(name):
    w = make_workload(name, device="cuda")
    flag = pkv.new_error_flag("cuda")
    out = _run(w, flag=flag)
    assert pkv.check_error(flag) == 0
    rng = np.random.default_rng(77)
    seqs = np.sort(rng.choice(w.spec.num_seqs, size=24, replace=False))
    expect, _, _ = oracle_after_append(w, seqs)
    assert_attention_close(out[torch.as_tensor(seqs, device="cuda")], expect, name)
    plain = pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                 w.max_context_len, scale=w.scale)
    assert torch.allclose(out.float(), plain.float(), atol=2e-3, rtol=1e-2)


def test_prefix_waits_for_work_queued_before_the_call():
    # The prefix kernel runs on a stream of the library's own; it must start only
    # after everything queued on the caller's stream before the call.  Here the
    # caller's stream spins for a while and then rewrites q: a prefix that did
    # not wait would attend with the old q.
    w = _make("bs16_g4_2groups")
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    torch.manual_seed(5)
    q_new = torch.randn_like(w.q, dtype=torch.float32).to(w.q.dtype)
    torch.cuda.synchronize()
    torch.cuda._sleep(20_000_000)
    w.q.copy_(q_new)
    out = _run(w, append=False)
    expect, _, _ = oracle_after_append(w)   # the oracle reads the new q
    assert_attention_close(out, expect, "prefix after queued work")


def test_caller_stream_work_after_the_call_sees_the_prefix():
    # Work the caller queues after the call (here a copy of the output) must see
    # the prefix partials merged, on the caller's own non-default stream.
    w = _make("bs32_g4_4groups")
    expect, _, _ = oracle_after_append(w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = _run(w)
        copy = out.clone()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert_attention_close(copy, expect, "caller stream")
