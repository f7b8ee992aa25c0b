"""The bench's algorithmic byte counts (the roofline numerator) against closed forms.

The KV bytes of one attention layer are 2 (K and V) x tokens x H_kv x d x
bytes per element ([inference] "KV Cache 的显存计算": 2·L·H·d·S·B·bytes, here
for one layer); queries and outputs add 2 x B x q_len x H_q x d x 2, the block
table 4 bytes per page read and the context lengths 4 bytes per sequence.  With
shared prefixes the prefix pages count once per group (unique physical slots),
which these tests compute from the group metadata instead of the block tables.
"""
import pytest
import torch

import bench
from workloads import make_workload


def _closed_form(w, q_len, kv_bytes, unique_tokens):
    s = w.spec
    lens = w.context_lens.long()
    pages = int(((lens + s.block_size - 1) // s.block_size).sum())
    kv = 2 * unique_tokens * s.num_kv_heads * s.head_dim * kv_bytes
    qo = 2 * s.num_seqs * q_len * s.num_q_heads * s.head_dim * 2
    return kv, kv + qo + 4 * pages + 4 * s.num_seqs


@pytest.mark.parametrize("q_len,kv_bytes", [(1, 2), (4, 2), (1, 1)])
def test_plain_workload_counts_every_context_token_once(q_len, kv_bytes):
    w = make_workload("c1", with_values=False)
    tokens = int(w.context_lens.sum())
    kv, decode = _closed_form(w, q_len, kv_bytes, tokens)
    got = bench.step_bytes(w, q_len, kv_bytes)
    assert got["kv_unique"] == kv
    assert got["decode"] == decode
    assert got["decode_logical"] == decode  # nothing shared: logical == unique
    s = w.spec
    assert got["flops"] == 4 * tokens * q_len * s.num_q_heads * s.head_dim
    assert got["tokens"] == s.num_seqs * q_len


def test_uniform_contexts_match_the_kv_size_formula():
    # every sequence at the same length L: KV = 2 * B * L * H_kv * d * 2
    w = make_workload("c3", with_values=False, num_seqs=4, lengths=("const", 1000),
                      max_len_cap=1024)
    s = w.spec
    assert torch.all(w.context_lens == 1000)
    got = bench.step_bytes(w)
    assert got["kv_unique"] == 2 * s.num_seqs * 1000 * s.num_kv_heads * s.head_dim * 2


def test_shared_prefix_pages_count_once_per_group():
    w = make_workload("c5", with_values=False, num_seqs=8, shared_prefix_groups=2,
                      lengths=("prefix_lognormal", 256, 64, 1.0, 1024), max_len_cap=1024)
    gs = w.group_start.long().tolist()
    gp = w.group_prefix_len.long().tolist()
    lens = w.context_lens.long().tolist()
    prefix_once = sum(gp)
    suffixes = sum(lens[b] - gp[g] for g in range(len(gp)) for b in range(gs[g], gs[g + 1]))
    kv, decode = _closed_form(w, 1, 2, prefix_once + suffixes)
    got = bench.step_bytes(w)
    assert got["kv_unique"] == kv
    assert got["decode"] == decode
    logical_kv = 2 * sum(lens) * w.spec.num_kv_heads * w.spec.head_dim * 2
    assert got["decode_logical"] - got["decode"] == logical_kv - kv > 0


@pytest.mark.parametrize("argv,what", [
    (["--config", "c5", "--splits", "4"], "--splits does not apply"),
    (["--config", "c5_bs32", "--splits", "12"], "--splits does not apply"),
    (["--splits", "4"], "--splits does not apply"),  # the default run includes c5
    (["--config", "c5", "--kv", "fp8"], "--kv fp8 times the plain decode path only"),
    (["--config", "c3", "--kv", "fp8", "--q-len", "4"], "--kv fp8 times the plain decode path only"),
    (["--config", "c3", "--q-len", "4", "--splits", "2"], "--splits does not apply to the multi-query"),
])
def test_bench_refuses_flags_a_step_cannot_honour(argv, what, capsys):
    """Refused on the host before any GPU work, so a line is never labelled with
    a split count or cache type that the timed step did not use."""
    with pytest.raises(SystemExit) as e:
        bench.main(argv)
    assert e.value.code == 2
    assert what in capsys.readouterr().err


@pytest.mark.parametrize("argv", [
    ["--config", "c5", "--splits", "4", "--no-prefix-sharing"],
    ["--config", "c3", "--splits", "4"],
    ["--config", "c3", "--kv", "fp8"],
    ["--config", "c5", "--kv", "fp8", "--no-prefix-sharing"],
    ["--config", "c5", "--q-len", "4"],
])
def test_bench_accepts_flags_the_step_honours(argv):
    args = _parse(argv)  # main() checks the flags before it would start the run
    assert args.config == argv[1]


def _parse(argv):
    """bench.main's parsing and checks, with the run itself replaced."""
    captured = {}

    def fake_run(args):
        captured["args"] = args

    old_gpu, old_ref = bench.run_gpu, bench.run_reference
    bench.run_gpu = bench.run_reference = fake_run
    try:
        bench.main(argv)
    finally:
        bench.run_gpu, bench.run_reference = old_gpu, old_ref
    return captured["args"]


def test_reference_arm_prints_the_contract_line():
    """The oracle arm (`--impl reference`) runs on the host cores and prints one
    JSON line with the keys the driver reads, on the arm's own metric and unit.
    It runs in a process of its own: the oracle's OpenMP threads must not live on
    in this one, whose later tests fork."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--config", "c1", "--steps", "3", "--warmup", "3", "--ref-seconds", "2"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "c1"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
