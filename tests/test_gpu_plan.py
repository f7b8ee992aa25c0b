"""The automatic split plan's choices on a 152-SM GB300 for the measured workloads.

The plan takes, among partitions of 256 to 2048 tokens, the count with the
least (waves of resident CTAs, rounded up) x (partition tokens + a fixed
start), preferring counts whose CTAs fill at least one wave.  These are the
counts the measured numbers were taken with; a change to the rule shows here.
"""
import pytest
import torch

import paged_kv_cache_164_gb300 as pkv
from workloads import make_workload

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _splits(name, kv="16bit", **kw):
    w = make_workload(name, with_values=False, **kw)
    s = w.spec
    return pkv.decode_num_splits(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                 s.block_size, w.max_context_len, kv=kv)


@pytest.mark.skipif(not torch.cuda.is_available() or _sms() != 152,
                    reason="the expected counts are for 152 SMs")
@pytest.mark.parametrize("name,kv,expect", [
    ("c2", "16bit", 2),   # 2048 units: 2 partitions of 2016 tokens, 9 waves
    ("c3", "16bit", 3),   # 256 units x 3 = 768 CTAs, 1.68 waves of 456
    ("c4", "16bit", 64),  # partitions of 2048 tokens at up to 131072
    ("c5", "16bit", 8),   # the suffix plan of the shared-prefix path
    ("c3", "fp8", 4),     # 2 would leave 0.84 of a wave of 608: 4 fill it
    ("c4", "fp8", 66),
])
def test_plan_counts(name, kv, expect):
    assert _splits(name, kv) == expect


def test_small_batches_split_finely():
    # 8 units cannot fill a wave at any count: the shortest partitions (256 tokens)
    if not torch.cuda.is_available():
        pytest.skip("needs the device")
    assert _splits("c3", num_seqs=1, lengths=("const", 4096), max_len_cap=4096) == 16
