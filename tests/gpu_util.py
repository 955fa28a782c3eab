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


def half_ulp_bf16(x):
    """Half a unit in the last place of bf16 at magnitude |x| (8 significant
    bits: 2^(floor(log2|x|) - 8)); 2^-134 at zero."""
    return np.exp2(np.floor(np.log2(np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126))) - 8)


def o_tight_bound(o_ref, o_absv_ref, n_keys):
    """Per-element bound on |O - O_ref| for the bf16 forward, from its
    arithmetic, with o_absv_ref = P|V| (the oracle's output for |V|):
      * P is rounded to bf16 (8 significant bits, unit roundoff 2^-8) before
        P V while l sums the unrounded p: the error of O~/l is at most
        2^-8 sum_j P_ij |V_jk| = 2^-8 (P|V|)_ik;
      * S = Q K^T in fp32 from exact bf16 products (d terms): an absolute
        error of at most about 2^-13 relative in each p, which moves O by at
        most 2^-11 (P|V|);
      * the fp32 accumulation of O~ over n_keys keys: at most n_keys 2^-23
        (P|V|), a worst case far above its typical size;
      * O rounded to bf16: half an ulp of the computed value, whose magnitude
        is at most |O_ref| plus the terms above.
    The bound has no global max|V| term, so it is tight where |O| and P|V|
    are small: a wrongly masked or unmasked key, or P rounded the wrong way,
    shows."""
    coef = 2.0 ** -8 + 2.0 ** -11 + n_keys * 2.0 ** -23
    pre = coef * np.asarray(o_absv_ref, dtype=np.float64)
    return pre + half_ulp_bf16(np.abs(np.asarray(o_ref, dtype=np.float64)) + pre) + 2.0 ** -24


def bf16_rne(x):
    """float64 values rounded to bf16 (nearest even) and back, via fp32 (exact
    for the magnitudes here: an fp32 double rounding can only differ at a
    tie of the fp64 value, which the oracle's outputs do not produce in
    practice)."""
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16).to(
        torch.float64).numpy()


def o_report(got, o_ref, o_absv_ref, n_keys, label):
    """Checks O element by element against o_tight_bound and returns the
    figures the parity record keeps: max-abs error against the float64 oracle,
    the largest error as a fraction of the tight bound, the share of elements
    equal to the oracle rounded to bf16 and the largest distance from it in
    bf16 ulps.  Also appended to the JSON-lines file named by
    FA_PARITY_REPORT, when set."""
    import json
    import os
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(o_ref, dtype=np.float64)
    a = np.asarray(o_absv_ref, dtype=np.float64)
    sel = ~np.isnan(r)  # sampled heads: the oracle leaves the others NaN
    g, r, a = g[sel], r[sel], a[sel]
    bound = o_tight_bound(r, a, n_keys)
    err = np.abs(g - r)
    rb = bf16_rne(r)
    ulp = 2.0 * half_ulp_bf16(rb)
    rec = {"case": label, "o_max_abs": float(err.max()) if err.size else 0.0,
           "tight_ratio_max": float((err / bound).max()) if err.size else 0.0,
           "equal_to_bf16_oracle": float((g == rb).mean()) if err.size else 1.0,
           "max_ulps_from_bf16_oracle": float((np.abs(g - rb) / ulp).max()) if err.size else 0.0}
    path = os.environ.get("FA_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
    bad = err > bound
    assert not bad.any(), (f"{label}: {int(bad.sum())} O elements past the tight bound; worst |err| "
                           f"{err.max():.3e}, worst err/bound {rec['tight_ratio_max']:.2f}")
    return rec
