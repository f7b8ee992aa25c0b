"""Append (scatter) and block-table gather on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_164_gb300 as pkv
from workloads import bits, make_append_case, make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("shape", [(300, 40, 16, 4, 64), (257, 33, 32, 8, 128), (64, 4096, 16, 32, 128)])
def test_append_bit_exact(dtype, shape):
    nt, nb, bs, h, d = shape
    c = make_append_case(nt, nb, bs, h, d, dtype, seed=nt + nb, device="cuda")
    kc, vc = bits(c["k_cache"]).copy(), bits(c["v_cache"]).copy()
    assert oracle.append(kc, vc, bits(c["k_new"]), bits(c["v_new"]),
                         c["slot_mapping"].cpu().numpy()) == 0
    flag = pkv.new_error_flag("cuda")
    pkv.append(c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], c["slot_mapping"],
               err_flag=flag)
    assert pkv.check_error(flag) == 0
    assert np.array_equal(bits(c["k_cache"]), kc)
    assert np.array_equal(bits(c["v_cache"]), vc)


def test_append_workload_new_tokens():
    w = make_workload("c5_bs32", num_seqs=16, lengths=("prefix_lognormal", 64, 40, 1.0, 400),
                      max_len_cap=512, shared_prefix_groups=2, device="cuda", poison=True)
    kc, vc = bits(w.k_cache).copy(), bits(w.v_cache).copy()
    oracle.append(kc, vc, bits(w.k_new), bits(w.v_new), w.slot_mapping.cpu().numpy())
    pkv.append(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    torch.cuda.synchronize()
    assert np.array_equal(bits(w.k_cache), kc) and np.array_equal(bits(w.v_cache), vc)


def test_append_slot_beyond_pool_is_flagged_and_skipped():
    c = make_append_case(20, 4, 16, 2, 64, "bf16", seed=9, pad_fraction=0.2, device="cuda")
    slots = c["slot_mapping"].clone()
    bad = int((slots >= 0).nonzero()[0])
    slots[bad] = 4 * 16 + 5
    kc, vc = bits(c["k_cache"]).copy(), bits(c["v_cache"]).copy()
    assert oracle.append(kc, vc, bits(c["k_new"]), bits(c["v_new"]), slots.cpu().numpy()) == -2
    flag = pkv.new_error_flag("cuda")
    pkv.append(c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], slots, err_flag=flag)
    assert pkv.check_error(flag) == pkv.EFLAG_SLOT
    assert np.array_equal(bits(c["k_cache"]), kc) and np.array_equal(bits(c["v_cache"]), vc)


@pytest.mark.parametrize("name", ["c1", "c5_bs32"])
def test_gather_bit_exact(name):
    kw = {} if name == "c1" else dict(num_seqs=8, lengths=("prefix_lognormal", 64, 40, 1.0, 400),
                                       max_len_cap=512, shared_prefix_groups=2)
    w = make_workload(name, device="cuda", **kw)
    mcl = w.max_context_len
    flag = pkv.new_error_flag("cuda")
    k_out, v_out = pkv.gather(w.k_cache, w.v_cache, w.block_tables, w.context_lens, mcl,
                              err_flag=flag)
    assert pkv.check_error(flag) == 0
    kc, vc = bits(w.k_cache), bits(w.v_cache)
    ko, vo = bits(k_out), bits(v_out)
    bt = w.block_tables.cpu().numpy()
    for b in range(w.spec.num_seqs):
        n = int(w.context_lens[b])
        for g in range(w.spec.num_kv_heads):
            ek, ev = oracle.gather_kv(kc, vc, bt, n, b, g)
            assert np.array_equal(ko[b, :n, g], ek) and np.array_equal(vo[b, :n, g], ev)
        assert np.all(ko[b, n:] == 0) and np.all(vo[b, n:] == 0)  # rows past n untouched


def test_gather_bad_block_id_is_flagged():
    w = make_workload("c1", device="cuda")
    bt = w.block_tables.clone()
    bt[1, 2] = w.num_blocks + 3
    flag = pkv.new_error_flag("cuda")
    pkv.gather(w.k_cache, w.v_cache, bt, w.context_lens, w.max_context_len, err_flag=flag)
    assert pkv.check_error(flag) == pkv.EFLAG_BLOCK_ID
