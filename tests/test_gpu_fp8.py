"""E4M3 (FP8) KV cache: quantising append and decode attention vs the oracle.

The append must store exactly the codes the oracle's quantiser gives (bit for
bit); decode over an E4M3 cache must match the oracle's attention over the
values the codes stand for (code * scale).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_164_gb300 as pkv
from helpers import assert_attention_close
from workloads import (bits, make_append_case, make_fp8_codes, make_workload, to_head_major)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs", [16, 64])
@pytest.mark.parametrize("scales", [(0.0123, 0.0311), (0.004, 0.5)])   # the first saturates some
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_quantising_append_matches_oracle_codes(dtype, scales, bs):
    c = make_append_case(200, 16, bs, 8, 128, dtype, seed=bs + 7, device="cuda")
    k_scale, v_scale = scales
    shape = (16, bs, 8, 128)
    kc = torch.full(shape, 0x5A, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    flag = pkv.new_error_flag("cuda")
    pkv.append_fp8(c["k_new"], c["v_new"], kc, vc, c["slot_mapping"], k_scale, v_scale,
                   err_flag=flag)
    assert pkv.check_error(flag) == 0
    ko = np.full(shape, 0x5A, dtype=np.uint8)
    vo = ko.copy()
    assert oracle.append_fp8(ko, vo, bits(c["k_new"]), bits(c["v_new"]),
                             c["slot_mapping"].cpu().numpy(), k_scale, v_scale, dtype) == 0
    assert np.array_equal(kc.cpu().numpy(), ko)
    assert np.array_equal(vc.cpu().numpy(), vo)
    # the head-major cache holds the same codes, permuted
    kh = torch.full((16, 8, bs, 128), 0x5A, dtype=torch.uint8, device="cuda")
    vh = kh.clone()
    pkv.append_fp8(c["k_new"], c["v_new"], kh, vh, c["slot_mapping"], k_scale, v_scale,
                   layout="hnd")
    assert torch.equal(kh, to_head_major(kc)) and torch.equal(vh, to_head_major(vc))


def _fp8_workload(case, k_scale, v_scale):
    """A workload whose 16-bit cache is quantised by the oracle (NaN in unused slots
    becomes the NaN code), with its new tokens appended by both sides."""
    name = case.pop("name")
    w = make_workload(name, device="cuda", poison=True, **case)
    k0 = oracle.encode_e4m3(w.k_cache.float().cpu().numpy() / np.float32(k_scale))
    v0 = oracle.encode_e4m3(w.v_cache.float().cpu().numpy() / np.float32(v_scale))
    kq, vq = k0.copy(), v0.copy()
    slots = w.slot_mapping.cpu().numpy()
    assert oracle.append_fp8(kq, vq, bits(w.k_new), bits(w.v_new), slots, k_scale, v_scale,
                             w.spec.dtype) == 0
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    pkv.append_fp8(w.k_new, w.v_new, kc, vc, w.slot_mapping, k_scale, v_scale)
    assert np.array_equal(kc.cpu().numpy(), kq)
    return w, kq, vq, kc, vc


CASES = {
    "gqa8_bf16": dict(name="c3", num_seqs=6, lengths=("uniform", 30, 1500), max_len_cap=1536,
                      seed=91),
    "mha_fp16": dict(name="c2", num_seqs=5, num_q_heads=8, num_kv_heads=8,
                     lengths=("uniform", 1, 700), max_len_cap=768, seed=92),
    "gqa4_bf16_bs32": dict(name="c5_bs32", num_seqs=7, shared_prefix_groups=0,
                           lengths=("uniform", 40, 900), max_len_cap=960, seed=93),
    "gqa16_fp16": dict(name="c3", num_seqs=3, num_q_heads=32, num_kv_heads=2, dtype="fp16",
                       lengths=("uniform", 100, 600), max_len_cap=640, seed=94),
}


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("key", sorted(CASES))
def test_fp8_decode_matches_oracle(key, splits):
    k_scale, v_scale = 5.0 / 448, 4.5 / 448
    w, kq, vq, kc, vc = _fp8_workload(dict(CASES[key]), k_scale, v_scale)
    expect = oracle.decode_attention_fp8(bits(w.q), kq, vq, w.block_tables.cpu().numpy(),
                                         w.context_lens.cpu().numpy(), w.scale, k_scale, v_scale,
                                         w.spec.dtype)
    flag = pkv.new_error_flag("cuda")
    out = pkv.decode_attention_fp8(w.q, kc, vc, w.block_tables, w.context_lens,
                                   w.max_context_len, k_scale, v_scale, scale=w.scale,
                                   num_splits=splits, err_flag=flag)
    assert pkv.check_error(flag) == 0
    assert_attention_close(out, expect, f"{key} splits={splits}")


def test_fp8_decode_on_head_major_cache_with_128_token_pages():
    k_scale, v_scale = 5.0 / 448, 4.5 / 448
    w, kq, vq, kc, vc = _fp8_workload(dict(CASES["gqa8_bf16"], block_size=128), k_scale, v_scale)
    expect = oracle.decode_attention_fp8(bits(w.q), kq, vq, w.block_tables.cpu().numpy(),
                                         w.context_lens.cpu().numpy(), w.scale, k_scale, v_scale,
                                         w.spec.dtype)
    out = pkv.decode_attention_fp8(w.q, to_head_major(kc), to_head_major(vc), w.block_tables,
                                   w.context_lens, w.max_context_len, k_scale, v_scale,
                                   scale=w.scale, layout="hnd")
    assert_attention_close(out, expect, "fp8 head-major bs128")


def test_fp8_full_size_llama70b_layer_sampled():
    w = make_workload("c3", device="cuda", with_values=False)
    s = w.spec
    kc = make_fp8_codes((w.num_blocks, s.block_size, s.num_kv_heads, s.head_dim), seed=95,
                        device="cuda")
    vc = make_fp8_codes(kc.shape, seed=96, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(97)
    q = torch.randn((s.num_seqs, s.num_q_heads, s.head_dim), generator=g, device="cuda",
                    dtype=torch.float32).to(torch.bfloat16)
    k_scale, v_scale = 0.37, 0.21
    flag = pkv.new_error_flag("cuda")
    out = pkv.decode_attention_fp8(q, kc, vc, w.block_tables, w.context_lens, w.max_context_len,
                                   k_scale, v_scale, err_flag=flag)
    assert pkv.check_error(flag) == 0
    seqs = np.array([0, 13, 31])
    expect = oracle.decode_attention_fp8(bits(q)[seqs], kc.cpu().numpy(), vc.cpu().numpy(),
                                         w.block_tables.cpu().numpy()[seqs],
                                         w.context_lens.cpu().numpy()[seqs],
                                         1.0 / np.sqrt(s.head_dim), k_scale, v_scale, "bf16")
    assert_attention_close(out[torch.as_tensor(seqs, device="cuda")], expect, "c3 fp8")
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_decode_subnormal_codes(dtype):
    # K and V hold only E4M3 subnormal codes (exponent field 0) and zeros, with
    # scales that make their values O(1): every product goes through the
    # conversion of subnormal codes, so one that lost them would be far off.
    w = make_workload("c3", device="cuda", with_values=False, num_seqs=3,
                      lengths=("uniform", 100, 420), max_len_cap=448, seed=98, dtype=dtype)
    s = w.spec
    kc = make_fp8_codes((w.num_blocks, s.block_size, s.num_kv_heads, s.head_dim), seed=99,
                        device="cuda", exponents=(0, 1))
    vc = make_fp8_codes(kc.shape, seed=100, device="cuda", exponents=(0, 1))
    g = torch.Generator(device="cuda").manual_seed(101)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    q = torch.randn((s.num_seqs, s.num_q_heads, s.head_dim), generator=g, device="cuda",
                    dtype=torch.float32).to(tdt)
    k_scale, v_scale = 64.0, 48.0     # code values m * 2^-9 become m / 8 and 3m / 32
    flag = pkv.new_error_flag("cuda")
    out = pkv.decode_attention_fp8(q, kc, vc, w.block_tables, w.context_lens, w.max_context_len,
                                   k_scale, v_scale, err_flag=flag)
    assert pkv.check_error(flag) == 0
    expect = oracle.decode_attention_fp8(bits(q), kc.cpu().numpy(), vc.cpu().numpy(),
                                         w.block_tables.cpu().numpy(), w.context_lens.cpu().numpy(),
                                         1.0 / np.sqrt(s.head_dim), k_scale, v_scale, dtype)
    assert_attention_close(out, expect, f"subnormal codes {dtype}")


@pytest.mark.parametrize("layout", ["nhd", "hnd"])
@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("key", sorted(CASES))
def test_fused_fp8_append_decode_matches_oracle_and_separate_append(key, splits, layout):
    # One launch: the decode kernel quantises each sequence's new token into the
    # slot of position n-1 (the same codes the oracle's quantiser gives, bit for
    # bit) and attends over the updated E4M3 cache.
    k_scale, v_scale = 5.0 / 448, 4.5 / 448
    case = dict(CASES[key])
    name = case.pop("name")
    w = make_workload(name, device="cuda", poison=True, **case)
    k0 = oracle.encode_e4m3(w.k_cache.float().cpu().numpy() / np.float32(k_scale))
    v0 = oracle.encode_e4m3(w.v_cache.float().cpu().numpy() / np.float32(v_scale))
    kq, vq = k0.copy(), v0.copy()
    assert oracle.append_fp8(kq, vq, bits(w.k_new), bits(w.v_new), w.slot_mapping.cpu().numpy(),
                             k_scale, v_scale, w.spec.dtype) == 0
    expect = oracle.decode_attention_fp8(bits(w.q), kq, vq, w.block_tables.cpu().numpy(),
                                         w.context_lens.cpu().numpy(), w.scale, k_scale, v_scale,
                                         w.spec.dtype)
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    if layout == "hnd":
        kc, vc = to_head_major(kc), to_head_major(vc)
    flag = pkv.new_error_flag("cuda")
    out = pkv.append_decode_attention_fp8(w.q, w.k_new, w.v_new, kc, vc, w.block_tables,
                                          w.context_lens, w.max_context_len, k_scale, v_scale,
                                          scale=w.scale, num_splits=splits, err_flag=flag,
                                          layout=layout)
    assert pkv.check_error(flag) == 0
    if layout == "hnd":
        kc, vc = kc.permute(0, 2, 1, 3).contiguous(), vc.permute(0, 2, 1, 3).contiguous()
    assert np.array_equal(kc.cpu().numpy(), kq) and np.array_equal(vc.cpu().numpy(), vq)
    assert_attention_close(out, expect, f"{key} splits={splits} {layout}")


def test_fused_fp8_full_size_llama70b_layer_sampled():
    # The E4M3 step the benchmark times on the Llama-70B layer (one fused launch,
    # automatic plan): every new token's codes bit for bit, sampled outputs
    # against the oracle.
    w = make_workload("c3", device="cuda", with_values=False)
    s = w.spec
    kc = make_fp8_codes((w.num_blocks, s.block_size, s.num_kv_heads, s.head_dim), seed=195,
                        device="cuda")
    vc = make_fp8_codes(kc.shape, seed=196, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(197)
    q, k_new, v_new = (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32)
                       .to(torch.bfloat16)
                       for shape in ((s.num_seqs, s.num_q_heads, s.head_dim),
                                     (s.num_seqs, s.num_kv_heads, s.head_dim),
                                     (s.num_seqs, s.num_kv_heads, s.head_dim)))
    k_scale, v_scale = 4.0 / 448, 3.5 / 448
    kq, vq = kc.cpu().numpy(), vc.cpu().numpy()
    assert oracle.append_fp8(kq, vq, bits(k_new), bits(v_new), w.slot_mapping.cpu().numpy(),
                             k_scale, v_scale, "bf16") == 0
    flag = pkv.new_error_flag("cuda")
    out = pkv.append_decode_attention_fp8(q, k_new, v_new, kc, vc, w.block_tables,
                                          w.context_lens, w.max_context_len, k_scale, v_scale,
                                          err_flag=flag)
    assert pkv.check_error(flag) == 0
    assert np.array_equal(kc.cpu().numpy(), kq) and np.array_equal(vc.cpu().numpy(), vq)
    seqs = np.array([0, 17, 31])
    expect = oracle.decode_attention_fp8(bits(q)[seqs], kq, vq, w.block_tables.cpu().numpy()[seqs],
                                         w.context_lens.cpu().numpy()[seqs],
                                         1.0 / np.sqrt(s.head_dim), k_scale, v_scale, "bf16")
    assert_attention_close(out[torch.as_tensor(seqs, device="cuda")], expect, "c3 fp8 fused")
    assert torch.isfinite(out).all()


def test_fused_fp8_append_skips_and_flags_a_bad_last_block():
    # A sequence whose last block id is out of range: flagged, its new token
    # not stored, every other sequence's token stored as usual.
    k_scale, v_scale = 5.0 / 448, 4.5 / 448
    case = dict(CASES["gqa8_bf16"])
    name = case.pop("name")
    w = make_workload(name, device="cuda", **case)
    kc = torch.from_numpy(oracle.encode_e4m3(w.k_cache.float().cpu().numpy() /
                                             np.float32(k_scale))).cuda()
    vc = torch.from_numpy(oracle.encode_e4m3(w.v_cache.float().cpu().numpy() /
                                             np.float32(v_scale))).cuda()
    before = kc.clone()
    bt = w.block_tables.clone()
    b, bs = 2, w.spec.block_size
    n = int(w.context_lens[b])
    bt[b, (n - 1) // bs] = w.num_blocks + 5   # out of range
    flag = pkv.new_error_flag("cuda")
    pkv.append_decode_attention_fp8(w.q, w.k_new, w.v_new, kc, vc, bt, w.context_lens,
                                    w.max_context_len, k_scale, v_scale, scale=w.scale,
                                    err_flag=flag)
    assert pkv.check_error(flag) & pkv.EFLAG_BLOCK_ID
    changed = (kc != before).any(dim=3).any(dim=2)
    slots = w.slot_mapping.cpu().tolist()
    expect_changed = {(s // bs, s % bs) for i, s in enumerate(slots) if i != b}
    got_changed = {tuple(x) for x in torch.nonzero(changed).cpu().tolist()}
    assert got_changed <= expect_changed
