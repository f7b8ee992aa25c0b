"""The small parity suite on the NaN-sentinel build (GPU).

The library built with -DPKV_DEBUG fills every shared-memory ring slot with
NaN bytes at the start and whenever its stage is released.  A kernel that
reads a slot before its copy lands, or reads a stage after releasing it (a
slip in an mbarrier phase), then writes NaN, which the oracle comparisons
reject.  This runs the small oracle-parity cases of the decode, multi-query,
shared-prefix, E4M3, layout and fuzz suites against that build, in a child
process that loads it in place of the normal one.
"""
import os
import subprocess
import sys

import pytest

from paged_kv_cache_164_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUITE = [
    "tests/test_gpu_decode.py::test_small_cases_all_splits",
    "tests/test_gpu_decode.py::test_edge_lengths",
    "tests/test_gpu_multi_query.py::test_multi_query_matches_oracle",
    "tests/test_gpu_prefix.py",
    "tests/test_gpu_fp8.py",
    "tests/test_gpu_layout.py",
    "tests/test_gpu_fused_graph.py",
    "tests/test_gpu_fuzz.py",
    "tests/test_gpu_debug_build.py::test_child_loaded_the_debug_build",
]


@pytest.mark.gpu
def test_small_parity_suite_on_the_nan_sentinel_build():
    lib = pkv_build.build(debug=True)
    env = dict(os.environ, PKV_LIBRARY=lib, PKV_EXPECT_DEBUG_BUILD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                        "-p", "no:cacheprovider", *SUITE],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail


@pytest.mark.gpu
@pytest.mark.skipif(os.environ.get("PKV_EXPECT_DEBUG_BUILD") != "1",
                    reason="runs inside the debug-build child process only")
def test_child_loaded_the_debug_build():
    import paged_kv_cache_164_gb300 as pkv
    assert pkv.load().pkv_debug_build() == 1
