"""pkv_merge against the oracle's log-sum-exp merge; device-side index errors."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_164_gb300 as pkv
from helpers import assert_attention_close, oracle_after_append
from workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_merge_matches_oracle(dtype, splits):
    g = torch.Generator().manual_seed(splits)
    b, h, d = 5, 6, 128
    po = torch.randn(b, h, splits, d, generator=g) * 0.5
    lse = torch.randn(b, h, splits, generator=g) * 3.0
    empty = torch.rand(b, h, splits, generator=g) < 0.3
    lse[empty] = float("-inf")
    lse[0, 0, :] = float("-inf")          # a row with every split empty
    expect = oracle.merge_lse(po.double().numpy(), lse.double().numpy())
    out = pkv.merge(po.cuda(), lse.cuda(), out_dtype=dtype)
    assert_attention_close(out, expect, f"merge {splits}")
    assert torch.all(out[0, 0] == 0)


def test_bad_block_id_is_flagged_not_faulted():
    w = make_workload("c3", num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=64,
                      lengths=("fixed", (100, 50, 70)), max_len_cap=128, pool="free_list",
                      pool_slack=0.3, seed=3, device="cuda")
    bt = w.block_tables.clone()
    bt[1, 1] = w.num_blocks + 1000
    bt[2, 0] = -5
    flag = pkv.new_error_flag("cuda")
    pkv.decode_attention(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.max_context_len,
                         err_flag=flag)
    assert pkv.check_error(flag) == pkv.EFLAG_BLOCK_ID
    # the library stays usable and correct afterwards
    expect, _, _ = oracle_after_append(w)
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                               w.max_context_len)
    assert_attention_close(out, expect, "after error")


def test_context_beyond_capacity_is_flagged():
    w = make_workload("c1", device="cuda")
    cl = w.context_lens.clone()
    cl[0] = w.max_blocks_per_seq * w.spec.block_size + 1
    flag = pkv.new_error_flag("cuda")
    pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, cl, int(cl.max()),
                         err_flag=flag)
    assert pkv.check_error(flag) & pkv.EFLAG_CONTEXT_LEN
    flag.zero_()
    # a context longer than the declared max_context_len is flagged too
    pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 40,
                         err_flag=flag)
    assert pkv.check_error(flag) & pkv.EFLAG_CONTEXT_LEN


def test_workspace_too_small_is_rejected():
    w = make_workload("c1", device="cuda")
    need = pkv.workspace_size(2, 4, 2, 64, 16, w.max_context_len, 2)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                             w.max_context_len, num_splits=2, workspace=small)
    assert e.value.status == 3


def test_bounded_wait_expires_with_a_status_not_a_hang():
    import time
    flag = pkv.new_error_flag("cuda")
    t0 = time.perf_counter()
    pkv.selftest_wait_timeout(flag, limit_ns=20_000_000)
    assert pkv.check_error(flag) == pkv.EFLAG_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # the context is still usable afterwards
    w = make_workload("c1", device="cuda")
    expect, _, _ = oracle_after_append(w)
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    out = pkv.decode_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                               w.max_context_len, scale=w.scale)
    assert_attention_close(out, expect, "after timeout self-test")
