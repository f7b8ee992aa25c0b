"""Shared test helpers: tolerance checks against the oracle, oracle runs on workloads."""
import numpy as np
import torch

import oracle
from workloads import bits

# Parity gate for attention outputs, in allclose form:
#     |gpu - oracle| <= ATOL + RTOL * |oracle|        element by element.
# (Both bounds elementwise cannot hold for bf16 outputs: rounding alone is up to
# 2^-9 relative, which exceeds 2e-3 absolute once |out| > 1.)
ATOL = 2e-3
RTOL = 1e-2
# Tighter precision check: the error must stay within one unit in the last place
# of the output type at the oracle's value, plus a small accumulation allowance.
ACC_EPS = 2e-5
_MANTISSA_BITS = {torch.float16: 10, torch.bfloat16: 7, torch.float32: 23}
_MIN_EXP = {torch.float16: -14, torch.bfloat16: -126, torch.float32: -126}


def ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Spacing of the 16-bit output type at |x| (the subnormal spacing below the normals)."""
    mb = _MANTISSA_BITS[dtype]
    ax = np.maximum(np.abs(x), 2.0 ** _MIN_EXP[dtype])
    return 2.0 ** (np.floor(np.log2(ax)) - mb)


def assert_attention_close(got: torch.Tensor, expect: np.ndarray, what: str = ""):
    g = got.detach().float().cpu().double().numpy()
    assert g.shape == expect.shape, (g.shape, expect.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    err = np.abs(g - expect)
    gate = ATOL + RTOL * np.abs(expect)
    worst = float((err / gate).max()) if err.size else 0.0
    assert worst <= 1.0, (f"{what}: parity gate exceeded by x{worst:.3f} "
                          f"(max abs err {float(err.max()):.3e})")
    tight = ulp(expect, got.dtype) + ACC_EPS
    worst_t = float((err / tight).max()) if err.size else 0.0
    assert worst_t <= 1.0, (f"{what}: error above one output ulp + {ACC_EPS}: "
                            f"x{worst_t:.3f} (max abs err {float(err.max()):.3e})")
    if got.dtype == torch.float16:
        assert_strict_bounds(err, expect, what)
    return float(err.max()) if err.size else 0.0


# The stated bounds read literally, both at once, element by element:
#     |gpu - oracle| <= 2e-3   and   |gpu - oracle| / max(|oracle|, 1e-3) <= 1e-2.
# fp16 outputs can meet them: an fp16 value below 8 in magnitude is within half
# an ulp (<= 2^-9) of the exact result when correctly rounded, and attention
# outputs are convex combinations of N(0,1) values (below 8).  bf16 outputs
# cannot (half an ulp is 2^-9 relative, above 2e-3 absolute once |out| > 1),
# which is why the allclose form above is the gate for both types.
STRICT_ABS = 2e-3
STRICT_REL = 1e-2
STRICT_REL_FLOOR = 1e-3


def assert_strict_bounds(err: np.ndarray, expect: np.ndarray, what: str = ""):
    if not err.size:
        return
    rel = err / np.maximum(np.abs(expect), STRICT_REL_FLOOR)
    assert float(err.max()) <= STRICT_ABS, (
        f"{what}: max abs err {float(err.max()):.3e} above {STRICT_ABS}")
    assert float(rel.max()) <= STRICT_REL, (
        f"{what}: max rel err {float(rel.max()):.3e} above {STRICT_REL}")


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
