"""Plants mistakes in copies of the C oracle (on the CPU) and checks the pins catch them.

Each mutant is the oracle's source with one plausible slip — a dropped scale, a
wrong GQA head index, block and offset swapped, V read from the K cache, no
max subtraction, a dropped token, a missing normalisation, a wrong fp16
exponent bias or a wrong bf16 shift — compiled into a temporary directory.
The same independent references the pin tests use (library conversion, dense
torch attention, the dominant-key closed form) must reject every mutant, while
the unmodified source passes them.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import build as oracle_build
from oracle.reference import load_library
from workloads import bits, make_workload

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
