"""Helpers shared by the GPU parity tests: device copies of the seeded inputs
and the error measures the gates use."""
import numpy as np
import torch

# Gates (written once, used by every parity test).
O_MAX_ABS = 1e-2       # bf16 forward output, max |O - O_oracle|
L_MAX_ABS = 1e-3       # log-sum-exp, max |L - L_oracle|
GRAD_REL_FRO = 2e-2    # dQ, dK, dV: ||x - x_oracle||_F / ||x_oracle||_F
FP8_O_REL_FRO = 6e-2   # FP8 forward output vs exact attention on the unquantised inputs


def to_dev(*ts):
    return [t.to("cuda").contiguous() for t in ts]


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def max_abs(got, ref, mask_nan=True):
    g, r = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    if mask_nan:
        sel = ~np.isnan(r)
        g, r = g[sel], r[sel]
    return float(np.abs(g - r).max()) if g.size else 0.0


# Denominator floor for the relative Frobenius error, as an RMS per element.
# With a single key the softmax is constant, so the exact dQ and dK are zero
# and a purely relative measure is undefined; the floor (far below the
# O(0.1-1) size of any nonzero gradient entry here) turns the gate into an
# absolute one only in that degenerate case.
REL_FRO_FLOOR_RMS = 1e-3


def rel_fro(got, ref):
    g, r = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    sel = ~np.isnan(r)
    g, r = g[sel], r[sel]
    floor = REL_FRO_FLOOR_RMS * np.sqrt(max(r.size, 1))
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), floor))


def o_rounding_bound(o_ref, v):
    """Per-element bound on |O - O_ref| that follows from the kernel's
    arithmetic: P is rounded to bf16 before P V (relative 2^-9 per entry, and
    l is summed from the unrounded values: 2^-8 max|V| in total) and O is
    rounded to bf16 on output (half an ulp of |O|)."""
    import numpy as np
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_ref), 1e-30))) - 8)
    return half_ulp + 2.0 ** -8 * float(f64(v).__abs__().max()) + 1e-4
