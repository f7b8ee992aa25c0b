"""Shared test helpers: tolerance check against the oracle, oracle runs on workloads."""
import numpy as np
import torch

import oracle
from workloads import bits

# Attention tolerance: |gpu - oracle| <= ATOL and |gpu - oracle| / max(|oracle|, REL_FLOOR) <= RTOL
# element by element (the relative bound uses a floor so outputs near zero are judged
# on an absolute scale of RTOL * REL_FLOOR = 1e-5).
ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = 1e-3


def assert_attention_close(got: torch.Tensor, expect: np.ndarray, what: str = ""):
    g = got.detach().float().cpu().double().numpy()
    assert g.shape == expect.shape, (g.shape, expect.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    err = np.abs(g - expect)
    rel = err / np.maximum(np.abs(expect), REL_FLOOR)
    worst_abs = float(err.max()) if err.size else 0.0
    worst_rel = float(rel.max()) if rel.size else 0.0
    assert worst_abs <= ATOL and worst_rel <= RTOL, \
        f"{what}: max abs err {worst_abs:.3e}, max rel err {worst_rel:.3e}"
    return worst_abs, worst_rel


def oracle_after_append(w, seqs=None):
    """Oracle output for workload ``w`` after its append, optionally for a subset of sequences.

    Everything is computed on the host from the generated inputs: the oracle's own
    append into host copies of the caches, then the oracle's decode attention.
    """
    kc = bits(w.k_cache).copy()
    vc = bits(w.v_cache).copy()
    rc = oracle.append(kc, vc, bits(w.k_new), bits(w.v_new), w.slot_mapping.cpu().numpy())
    assert rc == 0
    q = bits(w.q)
    bt = w.block_tables.cpu().numpy()
    cl = w.context_lens.cpu().numpy()
    if seqs is not None:
        q, bt, cl = q[seqs], bt[seqs], cl[seqs]
    return oracle.decode_attention(q, kc, vc, bt, cl, w.scale, w.spec.dtype), kc, vc
