"""Parity at the workloads' full sizes, in the launch configuration the bench
uses: the GPU computes every head; the float64 oracle checks sampled heads
(each costs it seconds to tens of seconds).  Same gates as the small cases."""
import math

import pytest
import torch

import oracle
from exact_attention_76_gb300 import api, build, inputs
from tests.gpu_util import FP8_O_REL_FRO, GRAD_REL_FRO, L_MAX_ABS, O_MAX_ABS, f64, max_abs, o_report, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    yield
    assert api.fa_device_error() == 0


def _fwd_bwd_sampled(B, H, N, d, causal, seed, heads, label):
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = inputs.draw_bf16(B, H, N, d, seed)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = api.fa_fwd(qd, kd, vd, causal, scale)
    dq, dk, dv = api.fa_bwd(qd, kd, vd, o, lse, dod, causal, scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.forward(q, k, v, causal, scale, heads=heads)
    absv_ref, _ = oracle.forward(q, k, v.abs(), causal, scale, heads=heads)
    g_ref = oracle.backward(q, k, v, do, causal, scale, heads=heads)
    eo, el = max_abs(f64(o), o_ref), max_abs(f64(lse), l_ref)
    eg = [rel_fro(f64(g), r) for g, r in zip((dq, dk, dv), g_ref)]
    assert eo <= O_MAX_ABS, f"O max-abs {eo:.3e}"
    assert el <= L_MAX_ABS, f"L max-abs {el:.3e}"
    o_report(f64(o), o_ref, absv_ref, N, label)
    for name, e in zip(("dQ", "dK", "dV"), eg):
        assert e <= GRAD_REL_FRO, f"{name} rel-Frobenius {e:.3e}"


def test_long_causal_workload_sampled_heads():
    w = inputs.LONG_CAUSAL
    _fwd_bwd_sampled(w.B, w.H, w.N, w.d, w.causal, w.seed, heads=[(0, 0), (1, 15)], label=w.name)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192, 16384])
def test_fixed_token_sweep_sampled_head(N, causal, d):
    # every length of the fixed-16384-token sweep, in its own launch shape
    ws = {w.N: w for w in inputs.sweep_workloads(causal, d)}
    w = ws[N]
    _fwd_bwd_sampled(w.B, w.H, w.N, w.d, causal, w.seed, heads=[(w.B - 1, w.H - 1)], label=w.name)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_workload_sampled_heads(causal):
    w = inputs.FP8
    scale = w.scale
    q, k, v = inputs.draw_outlier_fp32(w.B, w.H, w.N, w.d, w.seed)
    q8, dsq = api.fa_fp8_quantize(q.cuda(), True)
    k8, dsk = api.fa_fp8_quantize(k.cuda(), True)
    v8, dsv = api.fa_fp8_quantize(v.cuda(), False)
    o, lse = api.fa_fwd_fp8(q8, k8, v8, dsq, dsk, dsv, causal, scale)
    torch.cuda.synchronize()
    heads = [(0, 0), (0, 11)]
    o_ref, _ = oracle.forward_fp8_reference(q, k, v, causal, scale, heads=heads)
    e = rel_fro(f64(o), o_ref)
    assert e <= FP8_O_REL_FRO, f"FP8 O rel-Frobenius {e:.3e}"
