"""Structure of the seeded synthetic workloads (CPU only, no values for the big ones)."""
import math

import pytest
import torch

from workloads import SPECS, make_workload


def _check_tables(w):
    bs = w.spec.block_size
    seen = {}
    for b in range(w.spec.num_seqs):
        n = int(w.context_lens[b])
        used = (n + bs - 1) // bs
        row = w.block_tables[b]
        assert torch.all(row[:used] >= 0) and torch.all(row[:used] < w.num_blocks)
        assert torch.all(row[used:] == -1)
        for blk in row[:used].tolist():
            seen.setdefault(blk, set()).add(b)
        # the new token's slot is position n - 1 of the sequence
        s = int(w.slot_mapping[b])
        assert s // bs == int(row[(n - 1) // bs]) and s % bs == (n - 1) % bs
    return seen


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5", "c5_bs32"])
def test_structure(name):
    w = make_workload(name, with_values=False)
    spec = SPECS[name]
    seen = _check_tables(w)
    shared = [b for b, users in seen.items() if len(users) > 1]
    assert len(shared) == w.shared_blocks
    lens = w.context_lens.long()
    if name == "c1":
        assert lens.tolist() == [38, 51] and w.num_blocks == 16
    if name == "c2":
        assert lens.min() >= 512 and lens.max() <= 4096
    if name == "c3":
        assert torch.all(lens == 4096) and w.num_blocks == 32 * 256
    if name == "c4":
        assert lens.min() >= 32768 and lens.max() <= 131072
    if name.startswith("c5"):
        assert lens.min() >= 2049 and lens.max() <= 16384
        prefix_pages = 2048 // spec.block_size
        for g in range(4):
            rows = w.block_tables[g * 64:(g + 1) * 64, :prefix_pages]
            assert torch.all(rows == rows[0])
        # new tokens never land in a shared prefix block
        blocks = (w.slot_mapping // spec.block_size).tolist()
        assert not set(blocks) & set(shared)
        # suffix median close to the lognormal median 1024
        med = float((lens - 2048).float().median())
        assert 700 < med < 1500


def test_deterministic_and_seeded():
    a = make_workload("c2", num_seqs=4, lengths=("uniform", 5, 90), max_len_cap=96)
    b = make_workload("c2", num_seqs=4, lengths=("uniform", 5, 90), max_len_cap=96)
    c = make_workload("c2", num_seqs=4, lengths=("uniform", 5, 90), max_len_cap=96, seed=77)
    for f in ("context_lens", "block_tables", "slot_mapping", "q", "k_cache"):
        assert torch.equal(getattr(a, f), getattr(b, f))
    assert not torch.equal(a.block_tables, c.block_tables)


def test_values_standard_normal_and_poison():
    w = make_workload("c2", num_seqs=4, lengths=("uniform", 5, 90), max_len_cap=96, poison=True)
    bs = w.spec.block_size
    for b in range(4):
        n = int(w.context_lens[b])
        blk = int(w.block_tables[b, (n - 1) // bs])
        assert torch.isnan(w.k_cache[blk, (n - 1) % bs]).all()   # new token slot, pre-append
        if (n - 1) % bs:
            assert torch.isfinite(w.k_cache[blk, (n - 2) % bs]).all()
    x = w.q.float()
    assert abs(float(x.mean())) < 0.1 and abs(float(x.std()) - 1.0) < 0.1
