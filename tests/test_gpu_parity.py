"""Parity of the CUDA path (through the C ABI) with the float64 oracle on the
same seeded inputs.  Gates: O max-abs <= 1e-2, L max-abs <= 1e-3, dQ/dK/dV
relative Frobenius <= 2e-2, FP8 O relative Frobenius <= 6e-2."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_76_gb300 import api, build, inputs
from tests.gpu_util import (FP8_O_REL_FRO, GRAD_REL_FRO, L_MAX_ABS, O_MAX_ABS, f64, max_abs, o_report,
                            rel_fro, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    yield
    assert api.fa_device_error() == 0


def run_fwd_bwd(q, k, v, do, causal, scale):
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = api.fa_fwd(qd, kd, vd, causal, scale)
    dq, dk, dv = api.fa_bwd(qd, kd, vd, o, lse, dod, causal, scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def check_fwd(o, lse, q, k, v, causal, scale, heads=None, label="fwd"):
    """The literal gates (O max-abs, L max-abs) and, element by element, the
    tight bound of the kernel's arithmetic (tests/gpu_util.o_tight_bound)."""
    o_ref, l_ref = oracle.forward(q, k, v, causal, scale, heads=heads)
    absv_ref, _ = oracle.forward(q, k, v.abs(), causal, scale, heads=heads)
    eo = max_abs(f64(o), o_ref)
    el = max_abs(f64(lse), l_ref)
    assert eo <= O_MAX_ABS, f"O max-abs {eo:.3e}"
    assert el <= L_MAX_ABS, f"L max-abs {el:.3e}"
    o_report(f64(o), o_ref, absv_ref, k.shape[2], label)
    return eo, el


def check_bwd(dq, dk, dv, q, k, v, do, causal, scale, heads=None):
    ref = oracle.backward(q, k, v, do, causal, scale, heads=heads)
    errs = [rel_fro(f64(g), r) for g, r in zip((dq, dk, dv), ref)]
    for name, e in zip(("dQ", "dK", "dV"), errs):
        assert e <= GRAD_REL_FRO, f"{name} rel-Frobenius {e:.3e}"
    return errs


# ---------------------------------------------------------------- small and ragged

SMALL = [
    # (B, H, N, d, causal)
    (1, 2, 128, 64, False),    # the tiny workload
    (1, 2, 128, 64, True),
    (1, 1, 256, 128, False),
    (1, 1, 256, 128, True),
    (2, 2, 384, 64, True),     # several tiles, odd number of 128-row tiles
    (1, 2, 1, 64, False),      # a single row
    (1, 2, 17, 128, True),     # ragged: one partial tile
    (1, 1, 130, 64, False),    # ragged tail after a full tile
    (1, 1, 130, 128, True),
    (2, 1, 333, 128, False),
    (1, 3, 600, 64, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_forward_backward_small(B, H, N, d, causal):
    q, k, v, do = inputs.draw_bf16(B, H, N, d, seed=N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = run_fwd_bwd(q, k, v, do, causal, scale)
    check_fwd(o, lse, q, k, v, causal, scale, label=f"small B{B} H{H} N{N} d{d} c{int(causal)}")
    check_bwd(dq, dk, dv, q, k, v, do, causal, scale)


def test_tiny_workload_fp32_draws_rounded():
    w = inputs.TINY
    q, k, v, do = inputs.make_bf16(w)
    o, lse, dq, dk, dv = run_fwd_bwd(q, k, v, do, w.causal, w.scale)
    check_fwd(o, lse, q, k, v, w.causal, w.scale)
    check_bwd(dq, dk, dv, q, k, v, do, w.causal, w.scale)


@pytest.mark.parametrize("causal", [False, True])
def test_gpt2_small_workload(causal):
    w = inputs.GPT2
    q, k, v, do = inputs.make_bf16(w)
    o, lse, dq, dk, dv = run_fwd_bwd(q, k, v, do, causal, w.scale)
    check_fwd(o, lse, q, k, v, causal, w.scale, label=f"gpt2small c{int(causal)}")
    check_bwd(dq, dk, dv, q, k, v, do, causal, w.scale)


def test_causal_first_row_equals_first_value_row():
    q, k, v, do = inputs.draw_bf16(1, 2, 256, 128, seed=5)
    o, lse, *_ = run_fwd_bwd(q, k, v, do, True, 1 / math.sqrt(128))
    # row 0 attends to key 0 only: O_0 = V_0 exactly (V_0 is already bf16)
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])


def test_large_logits_rescale_path():
    # Scaled-up queries and keys that grow block by block make the running max
    # jump by more than the rescale threshold between key blocks, which
    # exercises the conditional rescale of the output accumulator.  The
    # softmax is then very peaked, so the literal 1e-2 gate of the N(0,1)
    # workloads does not apply: the bound used here follows from the
    # arithmetic -- P is rounded to bf16 before P V (relative 2^-9 per entry,
    # and l is summed from the unrounded values: 2^-8 max|V| in total), and O
    # is rounded to bf16 on output (half an ulp of |O|).
    q, k, v, do = inputs.draw_bf16(1, 2, 512, 64, seed=9)
    q = (q.float() * 6).to(torch.bfloat16)
    grow = torch.repeat_interleave(torch.tensor([1.0, 1.6, 2.2, 2.8]), 128)[None, None, :, None]
    k = (k.float() * grow).to(torch.bfloat16)
    o, lse, dq, dk, dv = run_fwd_bwd(q, k, v, do, False, 0.125)
    o_ref, l_ref = oracle.forward(q, k, v, False, 0.125)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_ref), 1e-30))) - 8)
    bound = half_ulp + 2.0 ** -8 * float(v.float().abs().max()) + 1e-4
    assert np.all(np.abs(f64(o) - o_ref) <= bound)
    assert max_abs(f64(lse), l_ref) <= L_MAX_ABS
    check_bwd(dq, dk, dv, q, k, v, do, False, 0.125)


# ---------------------------------------------------------------- grouped-query attention

@pytest.mark.parametrize("H,Hkv,N,d,causal", [
    (4, 1, 256, 128, True),    # multi-query: every query head shares one K/V head
    (6, 2, 333, 64, False),    # ragged tail
    (8, 4, 512, 128, True),
    (4, 2, 130, 64, True),
    (8, 2, 1, 128, True),      # one key: every block is the last, all but one row past the end
    (8, 1, 17, 64, False),
])
def test_gqa_forward_backward(H, Hkv, N, d, causal):
    B = 2
    q, _, _, do = inputs.draw_bf16(B, H, N, d, seed=H * 100 + N)
    _, k, v, _ = inputs.draw_bf16(B, Hkv, N, d, seed=Hkv * 100 + N + 1)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = api.fa_fwd_gqa(qd, kd, vd, causal, scale)
    # With fa_bwd_gqa_workspace_size bytes these few key/value heads take the
    # split path (one CTA per query head, dK and dV added into accumulators);
    # with fa_bwd_workspace_size bytes the path that sums a group on chip.
    full = api.fa_bwd_gqa_workspace_size(B, H, Hkv, N, d)
    base = api.fa_bwd_workspace_size(B, H, N, d)
    assert full > base
    grads = {}
    for tag, nbytes in (("split", full), ("group", base)):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        grads[tag] = api.fa_bwd_gqa(qd, kd, vd, o, lse, dod, causal, scale, workspace=ws)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.forward_gqa(q, k, v, causal, scale)
    assert max_abs(f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(f64(lse), l_ref) <= L_MAX_ABS
    o_report(f64(o), o_ref, oracle.forward_gqa(q, k, v.abs(), causal, scale)[0], N,
             f"gqa H{H} Hkv{Hkv} N{N} d{d} c{int(causal)}")
    refs = oracle.backward_gqa(q, k, v, do, causal, scale)
    for tag, (dq, dk, dv) in grads.items():
        for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
            e = rel_fro(f64(got), ref)
            assert e <= GRAD_REL_FRO, f"{tag} {name} rel-Frobenius {e:.3e}"


# ---------------------------------------------------------------- more work items than SMs
# More (query-tile pair, head) items than the GPU has SMs, of unequal length
# under the causal mask and with idle second tiles in the last query block of
# every head (ragged N): the cases a schedule that reuses CTAs across items
# must get right, kept as parity cases for the block-per-item schedule.

MANY_ITEMS = [
    # (B, H, Hkv, N, d, causal): ceil(N / 256) * B * H items, all above 152
    (4, 40, 40, 600, 64, True),
    (2, 48, 12, 520, 128, False),
    (2, 48, 48, 777, 128, True),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", MANY_ITEMS)
def test_forward_backward_many_items(B, H, Hkv, N, d, causal):
    q, _, _, do = inputs.draw_bf16(B, H, N, d, seed=N + H)
    _, k, v, _ = inputs.draw_bf16(B, Hkv, N, d, seed=N + Hkv + 1)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = api.fa_fwd_gqa(qd, kd, vd, causal, scale)
    dq, dk, dv = api.fa_bwd_gqa(qd, kd, vd, o, lse, dod, causal, scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.forward_gqa(q, k, v, causal, scale)
    assert max_abs(f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(f64(lse), l_ref) <= L_MAX_ABS
    o_report(f64(o), o_ref, oracle.forward_gqa(q, k, v.abs(), causal, scale)[0], N,
             f"many-items B{B} H{H} Hkv{Hkv} N{N} d{d} c{int(causal)}")
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), oracle.backward_gqa(q, k, v, do, causal, scale)):
        e = rel_fro(f64(got), ref)
        assert e <= GRAD_REL_FRO, f"{name} rel-Frobenius {e:.3e}"


def test_window_many_items():
    B, H, N, d, window = 2, 40, 700, 128, 300  # 240 items
    q, k, v, _ = inputs.draw_bf16(B, H, N, d, seed=window + 1)
    scale = 1 / math.sqrt(d)
    qd, kd, vd = to_dev(q, k, v)
    o, lse = api.fa_fwd_window(qd, kd, vd, window, scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.forward_window(q, k, v, window, scale)
    o_report(f64(o), o_ref, oracle.forward_window(q, k, v.abs(), window, scale)[0], N,
             f"window-many-items B{B} H{H} N{N} d{d} w{window}")
    assert max_abs(f64(lse), l_ref) <= L_MAX_ABS


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_many_items(causal, d):
    # 3 * 64 = 192 items; against exact attention on the dequantised inputs
    orig, codes, deltas, o, lse, scale = _fp8_case(640, causal, B=1, H=64, d=d)
    deq = [oracle.dequantize_e4m3(c, dl) for c, dl in zip(codes, deltas)]
    o_deq, l_deq = oracle.forward(*deq, causal, scale)
    e = rel_fro(f64(o), o_deq)
    assert e <= FP8_O_REL_FRO, f"FP8 O rel-Frobenius vs dequantised inputs {e:.3e}"
    assert max_abs(f64(lse), l_deq) <= 2e-2


# ---------------------------------------------------------------- step by step

def test_preprocess_and_convert_steps():
    B, H, N, d = 2, 3, 200, 128
    q, k, v, do = inputs.draw_bf16(B, H, N, d, seed=11)
    o = v  # any bf16 tensor serves as O for the row-dot step
    od, dod = to_dev(o, do)
    D, acc = api.fa_bwd_preprocess(od, dod)
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(D), oracle.row_dot(o, do), rtol=1e-5, atol=1e-4)
    assert torch.count_nonzero(acc).item() == 0
    # convert: bf16(scale * acc), round to nearest even, bit for bit
    src = torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(3)).cuda()
    dq = api.fa_bwd_dq_convert(src, 0.37)
    torch.cuda.synchronize()
    assert torch.equal(dq.cpu(), (src.cpu() * 0.37).to(torch.bfloat16))


def test_backward_in_three_calls_matches_fa_bwd():
    B, H, N, d, causal, scale = 1, 2, 384, 128, True, 1 / math.sqrt(128)
    q, k, v, do = inputs.draw_bf16(B, H, N, d, seed=21)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = api.fa_fwd(qd, kd, vd, causal, scale)
    D, acc = api.fa_bwd_preprocess(o, dod)
    dk, dv = api.fa_bwd_main(qd, kd, vd, lse, dod, D, acc, causal, scale)
    dq = api.fa_bwd_dq_convert(acc, scale)
    torch.cuda.synchronize()
    check_bwd(dq, dk, dv, q, k, v, do, causal, scale)


# ---------------------------------------------------------------- FP8

def _fp8_case(N, causal, seed=4, B=1, H=2, d=128):
    q, k, v = inputs.draw_outlier_fp32(B, H, N, d, seed=seed)
    codes, deltas = [], []
    for t in (q, k, v):  # per-tensor e4m3 storage, made by the oracle's quantiser
        c, dl = oracle.quantize_e4m3_reference(t)
        codes.append(c)
        deltas.append(float(np.float32(dl)))
    scale = 1 / math.sqrt(d)
    q8, k8, v8 = (torch.from_numpy(c).cuda() for c in codes)
    dsc = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in deltas]
    o, lse = api.fa_fwd_fp8(q8, k8, v8, *dsc, causal, scale)
    torch.cuda.synchronize()
    return (q, k, v), codes, deltas, o, lse, scale


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [256, 1000])
def test_fp8_forward_kernel_error(causal, N, d):
    # Against exact attention on the dequantised e4m3 inputs: what remains is
    # the kernel's own error (P stored as e4m3, fp32 accumulation).
    orig, codes, deltas, o, lse, scale = _fp8_case(N, causal, d=d)
    deq = [oracle.dequantize_e4m3(c, dl) for c, dl in zip(codes, deltas)]
    o_deq, l_deq = oracle.forward(*deq, causal, scale)
    e = rel_fro(f64(o), o_deq)
    assert e <= FP8_O_REL_FRO, f"FP8 O rel-Frobenius vs dequantised inputs {e:.3e}"
    assert max_abs(f64(lse), l_deq) <= 2e-2


@pytest.mark.xfail(reason="per-tensor e4m3 storage of the x10-outlier inputs alone costs 7.7-8.5% relative "
                          "Frobenius error (measured on the CPU); needs incoherent processing of Q and K",
                   strict=False)
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_vs_unquantised_per_tensor_only(causal):
    orig, codes, deltas, o, lse, scale = _fp8_case(1000, causal)
    o_ref, _ = oracle.forward_fp8_reference(*orig, causal, scale)
    e = rel_fro(f64(o), o_ref)
    assert e <= FP8_O_REL_FRO, f"FP8 O rel-Frobenius vs unquantised inputs {e:.3e}"


# The FP8 gate (6e-2 relative Frobenius against exact attention on the
# unquantised inputs) is the d = 128 FP8 workload's.  At d = 64 a Hadamard
# rotation spreads an outlier over half as many coordinates, and e4m3 storage
# of the x10-outlier inputs alone already costs up to 6.8 % (measured in
# float64 on the oracle's own quantised inputs): there the GPU's total error is
# bounded by that storage error plus the kernel's own share, at most 2 %.
FP8_KERNEL_SHARE = 2e-2


def _fp8_unquantised_bound(q, k, v, causal, scale, d, rotate_qk, block_rows=None):
    if d == 128:
        return FP8_O_REL_FRO
    o_ref, _ = oracle.forward_fp8_reference(q, k, v, causal, scale)
    deq = []
    for t, rot, br in ((q, rotate_qk, block_rows[0] if block_rows else None),
                       (k, rotate_qk, block_rows[1] if block_rows else None),
                       (v, False, block_rows[2] if block_rows else None)):
        y = oracle.rotate_rows(t) if rot else f64(t)
        if br is None:
            c, dl = oracle.quantize_e4m3_reference(y)
            deq.append(oracle.dequantize_e4m3(c, float(np.float32(dl))))
        else:
            c, dl = oracle.quantize_e4m3_blocks_reference(y, br)
            deq.append(oracle.dequantize_e4m3_blocks(c, dl.astype(np.float32).astype(np.float64), br))
    o_q, _ = oracle.forward(*deq, causal, scale)
    return rel_fro(o_q, o_ref) + FP8_KERNEL_SHARE


def _e4m3_codes(t):
    return torch.from_numpy(np.clip(t, -448.0, 448.0).astype(np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def _near_boundary_ok(got, ref_codes, x, y, t_scale, hadamard):
    """A code may differ from the fp64 reference only where y / delta lies
    within the kernel's fp32 error of an e4m3 rounding boundary: 2e-6 relative
    (the scaling by 1 / delta), plus, with the rotation, the rounding of the fp32 transform
    -- log2(d) stages of additions whose partial sums are bounded by the row's
    l1 norm, then the 1/sqrt(d) scaling: (log2 d + 1) 2^-24 |x_row|_1 / sqrt(d)
    in y (t_scale converts y to y / delta)."""
    d = y.shape[-1]
    t = y * t_scale
    tol = 2e-6 * np.abs(t)
    if hadamard:
        l1 = np.abs(f64(x)).sum(axis=-1, keepdims=True)
        tol = tol + (np.log2(d) + 1) * 2.0 ** -24 * l1 / np.sqrt(d) * np.abs(t_scale)
    return (got == ref_codes) | (got == _e4m3_codes(t - tol)) | (got == _e4m3_codes(t + tol))


@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fp8_quantize_matches_reference(hadamard, d, dtype):
    # The code is an integer decided in floating point: the kernel rotates in
    # fp32 and the reference in fp64, so a code may differ only where y/delta
    # lies within the kernel's fp32 error of an e4m3 rounding boundary.
    x = inputs.draw_outlier_fp32(1, 2, 300, d, seed=7)[0].to(dtype)
    codes, dsc = api.fa_fp8_quantize(x.cuda(), hadamard)
    torch.cuda.synchronize()
    y = oracle.rotate_rows(x) if hadamard else f64(x)
    ref_codes, ref_delta = oracle.quantize_e4m3_reference(y)
    delta = float(dsc.item())
    assert abs(delta - ref_delta) <= 1e-6 * ref_delta
    got = codes.cpu().numpy()
    assert _near_boundary_ok(got, ref_codes, x, y, 1.0 / ref_delta, hadamard).all()
    assert (got == ref_codes).mean() > 0.999


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [256, 1000])
def test_fp8_forward_with_incoherent_processing(causal, N, d):
    # Q and K rotated by the Hadamard transform before per-tensor e4m3
    # storage (V as is), against exact attention on the unquantised inputs.
    B, H = 1, 2
    q, k, v = inputs.draw_outlier_fp32(B, H, N, d, seed=4)
    scale = 1 / math.sqrt(d)
    q8, dsq = api.fa_fp8_quantize(q.cuda(), True)
    k8, dsk = api.fa_fp8_quantize(k.cuda(), True)
    v8, dsv = api.fa_fp8_quantize(v.cuda(), False)
    o, lse = api.fa_fwd_fp8(q8, k8, v8, dsq, dsk, dsv, causal, scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.forward_fp8_reference(q, k, v, causal, scale)
    e = rel_fro(f64(o), o_ref)
    bound = _fp8_unquantised_bound(q, k, v, causal, scale, d, True)
    assert e <= bound, f"FP8 O rel-Frobenius vs unquantised inputs {e:.3e} (bound {bound:.3e})"


# ---------------------------------------------------------------- FP8, block quantisation

@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("block_rows,dtype", [(64, torch.float32), (128, torch.float32), (128, torch.bfloat16),
                                              (48, torch.bfloat16), (48, torch.float32), (200, torch.float32),
                                              (200, torch.bfloat16)])
def test_fp8_quantize_blocks_matches_reference(hadamard, d, block_rows, dtype):
    # Same decision rule as the per-tensor quantiser: codes may differ only where
    # y/delta lies within the kernel's fp32 error of an e4m3 rounding boundary.
    # Blocks of 48 rows end inside a warp's 32 rows; 200 rows take the two-pass
    # form (four rows in flight per warp), for both input types.
    x = inputs.draw_outlier_fp32(1, 3, 300, d, seed=8)[0]
    x = (x * torch.exp2(torch.arange(300, dtype=torch.float32) // 50 - 3.0)[None, None, :, None]).to(dtype)
    codes, dsc = api.fa_fp8_quantize_blocks(x.cuda(), hadamard, block_rows)
    torch.cuda.synchronize()
    y = oracle.rotate_rows(x) if hadamard else f64(x)
    ref_codes, ref_deltas = oracle.quantize_e4m3_blocks_reference(y, block_rows)
    got_d = dsc.cpu().numpy().astype(np.float64).reshape(ref_deltas.shape)
    np.testing.assert_allclose(got_d, ref_deltas, rtol=1e-6, atol=0)
    got = codes.cpu().numpy()
    inv = 1.0 / np.repeat(ref_deltas, block_rows, axis=-1)[..., :300, None]
    assert _near_boundary_ok(got, ref_codes, x, y, inv, hadamard).all()
    assert (got == ref_codes).mean() > 0.999


@pytest.mark.parametrize("block_rows,dtype", [(64, torch.float32), (128, torch.bfloat16)])
def test_fp8_quantize_blocks_many_blocks(block_rows, dtype):
    # Enough rotated blocks (1024 or 512 over 8 sequences) that every CTA of
    # the block kernel takes several, staging the next one's rows while it
    # transforms the current one; blocks differ in magnitude by up to 2^8.
    x = inputs.draw_outlier_fp32(1, 8, 8192, 128, seed=13)[0]
    x = (x * torch.exp2((torch.arange(8192) // 64 % 9).to(torch.float32) - 4.0)[None, None, :, None]).to(dtype)
    codes, dsc = api.fa_fp8_quantize_blocks(x.cuda(), True, block_rows)
    torch.cuda.synchronize()
    y = oracle.rotate_rows(x)
    ref_codes, ref_deltas = oracle.quantize_e4m3_blocks_reference(y, block_rows)
    got_d = dsc.cpu().numpy().astype(np.float64).reshape(ref_deltas.shape)
    np.testing.assert_allclose(got_d, ref_deltas, rtol=1e-6, atol=0)
    got = codes.cpu().numpy()
    inv = 1.0 / np.repeat(ref_deltas, block_rows, axis=-1)[..., None]
    assert _near_boundary_ok(got, ref_codes, x, y, inv, True).all()
    assert (got == ref_codes).mean() > 0.999


def test_fp8_quantize_back_to_back_calls():
    # Calls queued back to back on one stream: each call's codes kernel starts
    # while its max|y| kernel finishes and reads x before waiting for it, so a
    # missing wait or a stale maximum (another call's) would show here.
    xs = [(inputs.draw_outlier_fp32(1, 2, 300 + 37 * i, 128, seed=20 + i)[0] * 4.0 ** i).to(dt)
          for i, dt in enumerate((torch.float32, torch.bfloat16, torch.float32))]
    dev = [x.cuda() for x in xs]
    torch.cuda.synchronize()
    outs = [(x, had, api.fa_fp8_quantize(xd, had)) for x, xd in zip(xs, dev) for had in (False, True)]
    torch.cuda.synchronize()
    for x, had, (codes, dsc) in outs:
        y = oracle.rotate_rows(x) if had else f64(x)
        ref_codes, ref_delta = oracle.quantize_e4m3_reference(y)
        assert abs(float(dsc.item()) - ref_delta) <= 1e-6 * ref_delta
        got = codes.cpu().numpy()
        assert _near_boundary_ok(got, ref_codes, x, y, 1.0 / ref_delta, had).all()
        assert (got == ref_codes).mean() > 0.999


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_quantize_bf16_codes_exact(d):
    # bf16 input, no rotation: y / delta = 448 x / max|x| = 7 (a / b) 2^k with
    # a, b the 8-bit significands.  Such a ratio is either short enough to be
    # exact (an e4m3 value, or an e4m3 midpoint that rounds to even) or at
    # least 2^-33 relative away from every fp32 rounding boundary, farther than
    # the kernels' error (about 2^-47) and the float64 reference's, so every
    # code equals the reference's.  0.6-1.0 % of these codes are exact
    # midpoints; a quotient by the rounded fp32 delta turns 0.8 % of the codes
    # of seed 16 at d = 128 the other way.
    for seed in (7, 16):
        x = inputs.draw_outlier_fp32(1, 2, 300, d, seed=seed)[0].to(torch.bfloat16)
        y = f64(x)
        codes, _ = api.fa_fp8_quantize(x.cuda(), False)
        blocks, _ = api.fa_fp8_quantize_blocks(x.cuda(), False, 64)
        torch.cuda.synchronize()
        assert np.array_equal(codes.cpu().numpy(), oracle.quantize_e4m3_reference(y)[0])
        assert np.array_equal(blocks.cpu().numpy(), oracle.quantize_e4m3_blocks_reference(y, 64)[0])


@pytest.mark.parametrize("hadamard", [False, True])
def test_fp8_quantize_tiny_and_zero_scales(hadamard):
    # max|y| below 2^-100 (the kernels scale y by 2^100 before the product with
    # 448 / max|y|, which would overflow otherwise) and all-zero tensors and
    # blocks (delta = 1, every code 0), per tensor and per 64-row block.
    d = 128
    x = inputs.draw_outlier_fp32(1, 2, 320, d, seed=9)[0]
    y_of = (lambda t: oracle.rotate_rows(t)) if hadamard else f64
    for t in (x * 2.0 ** -110, torch.zeros_like(x)):
        codes, dsc = api.fa_fp8_quantize(t.cuda(), hadamard)
        torch.cuda.synchronize()
        y = y_of(t)
        ref_codes, ref_delta = oracle.quantize_e4m3_reference(y)
        assert abs(float(dsc.item()) - ref_delta) <= 1e-6 * ref_delta
        got = codes.cpu().numpy()
        assert _near_boundary_ok(got, ref_codes, t, y, 1.0 / ref_delta, hadamard).all()
        assert (got == ref_codes).mean() > 0.999
    f = torch.tensor([0.0, 2.0 ** -110, 1.0, 2.0 ** -60, 0.0])[torch.arange(320) // 64]
    t = x * f[None, None, :, None] + 0.0  # +0 zero blocks: a rotated zero's sign follows the butterflies
    codes, dsc = api.fa_fp8_quantize_blocks(t.cuda(), hadamard, 64)
    torch.cuda.synchronize()
    y = y_of(t)
    ref_codes, ref_deltas = oracle.quantize_e4m3_blocks_reference(y, 64)
    got_d = dsc.cpu().numpy().astype(np.float64).reshape(ref_deltas.shape)
    np.testing.assert_allclose(got_d, ref_deltas, rtol=1e-6, atol=0)
    assert np.all(got_d[..., [0, 4]] == 1.0)
    got = codes.cpu().numpy()
    assert np.all(got[..., :64, :] == 0) and np.all(got[..., 256:, :] == 0)
    inv = 1.0 / np.repeat(ref_deltas, 64, axis=-1)[..., None]
    assert _near_boundary_ok(got, ref_codes, t, y, inv, hadamard).all()
    assert (got == ref_codes).mean() > 0.999


def _block_scaled_inputs(B, H, N, d, seed):
    # outlier inputs whose 64-row blocks also differ in magnitude by up to 2^12
    q, k, v = inputs.draw_outlier_fp32(B, H, N, d, seed=seed)
    g = torch.Generator().manual_seed(seed + 100)
    out = []
    for t in (q, k, v):
        e = torch.randint(-12, 1, (B, H, -(-N // 64)), generator=g).to(torch.float32)
        f = torch.exp2(e).repeat_interleave(64, dim=-1)[..., :N, None]
        out.append(t * f if t is v else t * f.sqrt())
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [256, 1000])
def test_fp8_blocks_forward_kernel_error(causal, N, d):
    # Against exact attention on the dequantised block-quantised inputs: what
    # remains is the kernel's own error (P as e4m3, fp32 accumulation).
    B, H = 1, 2
    q, k, v = _block_scaled_inputs(B, H, N, d, seed=4)
    scale = 1 / math.sqrt(d)
    cq, dq = oracle.quantize_e4m3_blocks_reference(q, api.FP8_BLOCK_Q)
    ck, dk = oracle.quantize_e4m3_blocks_reference(k, api.FP8_BLOCK_KV)
    cv, dv = oracle.quantize_e4m3_blocks_reference(v, api.FP8_BLOCK_KV)
    dev = [torch.from_numpy(c).cuda() for c in (cq, ck, cv)]
    dsc = [torch.from_numpy(x.reshape(B * H, -1).astype(np.float32)).cuda() for x in (dq, dk, dv)]
    o, lse = api.fa_fwd_fp8_blocks(*dev, *dsc, causal, scale)
    torch.cuda.synchronize()
    deq = [oracle.dequantize_e4m3_blocks(c, x.astype(np.float32).astype(np.float64), r)
           for c, x, r in ((cq, dq, 128), (ck, dk, 64), (cv, dv, 64))]
    o_ref, l_ref = oracle.forward(*deq, causal, scale)
    e = rel_fro(f64(o), o_ref)
    assert e <= FP8_O_REL_FRO, f"block FP8 O rel-Frobenius vs dequantised inputs {e:.3e}"
    assert max_abs(f64(lse), l_ref) <= 2e-2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_blocks_forward_with_incoherent_processing(causal, d):
    # The whole FP8 path on the GPU: Hadamard-rotated Q and K and plain V stored
    # per block, against exact attention on the unquantised inputs.
    B, H, N = 1, 2, 1000
    q, k, v = inputs.draw_outlier_fp32(B, H, N, d, seed=4)
    scale = 1 / math.sqrt(d)
    q8, dsq = api.fa_fp8_quantize_blocks(q.cuda(), True, api.FP8_BLOCK_Q)
    k8, dsk = api.fa_fp8_quantize_blocks(k.cuda(), True, api.FP8_BLOCK_KV)
    v8, dsv = api.fa_fp8_quantize_blocks(v.cuda(), False, api.FP8_BLOCK_KV)
    o, lse = api.fa_fwd_fp8_blocks(q8, k8, v8, dsq, dsk, dsv, causal, scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.forward_fp8_reference(q, k, v, causal, scale)
    e = rel_fro(f64(o), o_ref)
    bound = _fp8_unquantised_bound(q, k, v, causal, scale, d, True,
                                   (api.FP8_BLOCK_Q, api.FP8_BLOCK_KV, api.FP8_BLOCK_KV))
    assert e <= bound, f"block FP8 O rel-Frobenius vs unquantised inputs {e:.3e} (bound {bound:.3e})"


# ---------------------------------------------------------------- sliding window

WINDOW_CASES = [
    # (B, H, Hkv, N, d, window)
    (1, 2, 2, 256, 64, 63),     # window edge inside a 64-key block
    (1, 2, 2, 256, 64, 64),
    (1, 2, 2, 256, 128, 1),     # each row sees only its own key
    (1, 4, 2, 1000, 128, 100),  # grouped queries, ragged tail
    (1, 2, 2, 1000, 128, 257),  # window spans tiles; the second tile starts later
    (2, 2, 1, 777, 64, 700),
    (1, 2, 2, 1000, 64, 257),   # d = 64: the second tile starts later, S issued ahead of the softmax
    (1, 4, 2, 2000, 64, 300),
]


@pytest.mark.parametrize("B,H,Hkv,N,d,window", WINDOW_CASES)
def test_window_forward_backward(B, H, Hkv, N, d, window):
    q, k, v, do = inputs.draw_bf16(B, H, N, d, seed=window)
    k, v = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = api.fa_fwd_window(qd, kd, vd, window, scale)
    dq, dk, dv = api.fa_bwd_window(qd, kd, vd, o, lse, dod, window, scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.forward_window(q, k, v, window, scale)
    # A row averages at most `window` values, so |O| is larger than under full
    # attention and its bf16 rounding alone can pass the 1e-2 of the N(0,1)
    # gate: O is checked element by element against the tight bound that
    # follows from the arithmetic (which is below 1e-2 wherever |O| < 2).
    o_report(f64(o), o_ref, oracle.forward_window(q, k, v.abs(), window, scale)[0], N,
             f"window B{B} H{H} Hkv{Hkv} N{N} d{d} w{window}")
    assert max_abs(f64(lse), l_ref) <= L_MAX_ABS
    refs = oracle.backward_window(q, k, v, do, window, scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
        e = rel_fro(f64(g), r)
        assert e <= GRAD_REL_FRO, f"{name} rel-Frobenius {e:.3e}"


def test_window_at_least_n_is_causal_bit_for_bit():
    q, k, v, do = to_dev(*inputs.draw_bf16(1, 2, 500, 128, seed=21))
    o1, l1 = api.fa_fwd(q, k, v, True, 0.1)
    o2, l2 = api.fa_fwd_window(q, k, v, 500, 0.1)
    dq1, dk1, dv1 = api.fa_bwd(q, k, v, o1, l1, do, True, 0.1)
    dq2, dk2, dv2 = api.fa_bwd_window(q, k, v, o2, l2, do, 10 ** 6, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # dQ sums fp32 contributions in an order that varies run to run
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max().item() <= 2e-3


def test_window_long_sequence_sampled_heads():
    B, H, N, d, window = 1, 4, 4096, 128, 512
    q, k, v, do = inputs.draw_bf16(B, H, N, d, seed=22)
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = api.fa_fwd_window(qd, kd, vd, window, scale)
    dq, dk, dv = api.fa_bwd_window(qd, kd, vd, o, lse, dod, window, scale)
    torch.cuda.synchronize()
    h = 3
    sl = slice(h, h + 1)
    o_ref, l_ref = oracle.forward_window(q[:, sl], k[:, sl], v[:, sl], window, scale)
    o_report(f64(o[:, sl]), o_ref, oracle.forward_window(q[:, sl], k[:, sl], v[:, sl].abs(), window, scale)[0], N,
             f"window-long N{N} w{window}")
    assert max_abs(f64(lse[:, sl]), l_ref) <= L_MAX_ABS
    refs = oracle.backward_window(q[:, sl], k[:, sl], v[:, sl], do[:, sl], window, scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq[:, sl], dk[:, sl], dv[:, sl]), refs):
        e = rel_fro(f64(g), r)
        assert e <= GRAD_REL_FRO, f"{name} rel-Frobenius {e:.3e}"


# ---------------------------------------------------------------- random configurations

def _random_config(seed):
    r = np.random.default_rng(1000 + seed)
    d = int(r.choice([64, 128]))
    Hkv = int(r.choice([1, 2, 3]))
    H = Hkv * int(r.choice([1, 2, 4]))
    N = int(r.choice([1, 2, 3, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 511, 640, 700]))
    mode = str(r.choice(["full", "causal", "window"]))
    window = int(r.integers(1, 2 * N + 2)) if mode == "window" else 0
    return int(r.integers(1, 3)), H, Hkv, N, d, mode, window


@pytest.mark.parametrize("seed", range(24))
def test_random_configurations(seed):
    # Seeded random shapes (ragged lengths down to one token, grouped heads,
    # both head sizes, full / causal / windowed) through the public entry
    # points, forward and backward, against the oracle.
    B, H, Hkv, N, d, mode, window = _random_config(seed)
    q, k, v, do = inputs.draw_bf16(B, H, N, d, seed=seed)
    k, v = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    if mode == "window":
        o, lse = api.fa_fwd_window(qd, kd, vd, window, scale)
        dq, dk, dv = api.fa_bwd_window(qd, kd, vd, o, lse, dod, window, scale)
        o_ref, l_ref = oracle.forward_window(q, k, v, window, scale)
        absv_ref = oracle.forward_window(q, k, v.abs(), window, scale)[0]
        refs = oracle.backward_window(q, k, v, do, window, scale)
    else:
        causal = mode == "causal"
        o, lse = api.fa_fwd_gqa(qd, kd, vd, causal, scale)
        dq, dk, dv = api.fa_bwd_gqa(qd, kd, vd, o, lse, dod, causal, scale)
        o_ref, l_ref = oracle.forward_gqa(q, k, v, causal, scale)
        absv_ref = oracle.forward_gqa(q, k, v.abs(), causal, scale)[0]
        refs = oracle.backward_gqa(q, k, v, do, causal, scale)
    torch.cuda.synchronize()
    # Element by element against the tight bound of the arithmetic (a row
    # under a short window averages few values, so |O| can be large enough
    # for bf16 output rounding alone to pass the 1e-2 of the N(0,1) gate).
    o_report(f64(o), o_ref, absv_ref, N, f"random seed{seed} ({B},{H},{Hkv},{N},{d},{mode},{window})")
    assert max_abs(f64(lse), l_ref) <= L_MAX_ABS
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
        e = rel_fro(f64(g), r)
        assert e <= GRAD_REL_FRO, f"{name} rel-Frobenius {e:.3e} ({B},{H},{Hkv},{N},{d},{mode},{window})"


# ---------------------------------------------------------------- decode

def _decode_case(B, H, Hkv, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, N, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, N, d), generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 63, 64, 1000, 5000])
@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (8, 2), (6, 2), (16, 1)])
def test_decode_matches_oracle(d, N, H, Hkv):
    B = 2
    q, k, v = _decode_case(B, H, Hkv, N, d, seed=N + H)
    scale = 1 / math.sqrt(d)
    o, lse = api.fa_decode(q.cuda(), k.cuda(), v.cuda(), scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.decode(q, k, v, scale)
    assert max_abs(f64(o), o_ref) <= O_MAX_ABS
    assert max_abs(f64(lse), l_ref) <= L_MAX_ABS


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(16, 8), (32, 8)])
def test_decode_running_max_raised_within_a_chunk(d, H, Hkv):
    # Keys whose scale grows along the cache (1 + 0.01 n) raise each head's
    # running maximum by more than the rescale threshold about every second
    # 128-key tile, and query scales that differ per head make the heads raise
    # at different tiles; B * Hkv = 32 key/value heads split the cache into
    # chunks of several tiles, so the rescale of the output accumulator inside
    # a chunk is exercised.  The softmax is peaked, so O is held to the bound
    # that follows from the arithmetic (bf16 P, relative 2^-9 per entry, and l
    # from the unrounded values: 2^-8 max|V| in all; half an ulp of |O| from
    # the bf16 output), as in the forward's rescale test.
    B, N = 4, 4096
    q, k, v = _decode_case(B, H, Hkv, N, d, seed=21 + H)
    k = (k.float() * (1.0 + 0.01 * torch.arange(N, dtype=torch.float32))[None, None, :, None]).to(torch.bfloat16)
    q = (q.float() * (0.5 + torch.arange(H, dtype=torch.float32) / H)[None, :, None]).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    o, lse = api.fa_decode(q.cuda(), k.cuda(), v.cuda(), scale)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.decode(q, k, v, scale)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(o_ref), 1e-30))) - 8)
    bound = half_ulp + 2.0 ** -8 * float(v.float().abs().max()) + 1e-4
    assert np.all(np.abs(f64(o) - o_ref) <= bound)
    assert max_abs(f64(lse), l_ref) <= L_MAX_ABS


def test_decode_long_cache_and_reused_workspace():
    # 32768 keys per head in many chunks; the oracle's row costs O(N d), so every
    # head is checked.  The same workspace serves two different calls.
    B, H, Hkv, N, d = 2, 16, 4, 32768, 128
    q, k, v = _decode_case(B, H, Hkv, N, d, seed=11)
    scale = 1 / math.sqrt(d)
    ws = torch.empty(api.fa_decode_workspace_size(B, H, Hkv, N, d), dtype=torch.uint8, device="cuda")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = api.fa_decode(qd, kd, vd, scale, workspace=ws)
    o2, l2 = api.fa_decode(qd[:, :, :], kd[:, :, : N // 3].contiguous(), vd[:, :, : N // 3].contiguous(), scale,
                           workspace=ws)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.decode(q, k, v, scale)
    assert max_abs(f64(o1), o_ref) <= O_MAX_ABS
    assert max_abs(f64(l1), l_ref) <= L_MAX_ABS
    o_ref2, l_ref2 = oracle.decode(q, k[:, :, : N // 3], v[:, :, : N // 3], scale)
    assert max_abs(f64(o2), o_ref2) <= O_MAX_ABS
    assert max_abs(f64(l2), l_ref2) <= L_MAX_ABS


def test_decode_equals_the_last_row_of_the_causal_forward():
    # the same bf16 inputs through both kernels: decode of the last token against
    # the whole cache is the forward's last causal row
    B, H, N, d = 1, 4, 777, 128
    q, k, v, _ = inputs.draw_bf16(B, H, N, d, seed=12)
    scale = 1 / math.sqrt(d)
    o_f, l_f = api.fa_fwd(q.cuda(), k.cuda(), v.cuda(), True, scale)
    o_d, l_d = api.fa_decode(q[:, :, -1].contiguous().cuda(), k.cuda(), v.cuda(), scale)
    torch.cuda.synchronize()
    assert (o_d.float() - o_f[:, :, -1].float()).abs().max().item() <= 2 * O_MAX_ABS
    assert (l_d - l_f[:, :, -1]).abs().max().item() <= 2 * L_MAX_ABS


def test_decode_argument_checks():
    q = torch.zeros(1, 3, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        api.fa_decode(q, k, k, 0.1)  # 3 query heads over 2 key/value heads
    with pytest.raises(RuntimeError):
        api.fa_decode(torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda"), k, k, 0.1,
                      workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))


# ---------------------------------------------------------------- errors and the timeout path

def test_timeout_path_reports_and_context_survives():
    assert api.fa_debug_wait_timeout(2000) == 0
    assert api.fa_device_error() == 5  # FA_ERR_TIMEOUT
    assert api.fa_device_error() == 0  # cleared
    q, k, v, do = inputs.draw_bf16(1, 1, 128, 64, seed=1)
    o, lse, *_ = run_fwd_bwd(q, k, v, do, False, 0.125)
    check_fwd(o, lse, q, k, v, False, 0.125)


def test_ex2_rate_measurement():
    # a rate per SM and clock: positive and below one result per lane of the
    # SM's four 32-lane sub-partitions
    rate = api.fa_measure_ex2_rate()
    assert 1.0 < rate <= 128.0


def test_python_argument_checks():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(TypeError):
        api.fa_fwd(q, q, q, False, 0.125)
    qb = torch.zeros(1, 1, 128, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError, match="FA_ERR_UNSUPPORTED"):
        api.fa_fwd(qb, qb, qb, False, 0.125)


# ---------------------------------------------------------------- FMA-pipe exp2

@pytest.mark.parametrize("degree,bound", [(2, 1.73e-3), (3, 7.5e-5)])
def test_exp2_polynomial_on_the_gpu(degree, bound):
    # The device polynomial against exact 2^x over the range it serves, and
    # against the host model of its float32 steps (tests/test_exp2_poly.py,
    # whose generator produced the coefficients) to one ulp.
    import importlib.util
    import os
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "exact_attention_76_gb300",
                        "csrc")
    spec = importlib.util.spec_from_file_location("exp2_minimax", os.path.join(csrc, "exp2_minimax.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    x = np.concatenate([np.linspace(-125.5, 127.0, 2_000_001), np.linspace(-1.0, 1.0, 100_001),
                        np.arange(-125, 128) + 0.5 - 1e-3]).astype(np.float32)
    y = f64(api.fa_debug_exp2_poly(torch.from_numpy(x).cuda(), degree))
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() <= bound, f"degree {degree}: max relative error {rel.max():.3e}"
    model = gen.eval_exp2_f32(x, gen.coefficients_f32(degree)).astype(np.float64)
    assert np.all(np.abs(y - model) <= np.spacing(np.abs(model).astype(np.float32)).astype(np.float64))
    # below the range the result stands in for zero
    tiny = f64(api.fa_debug_exp2_poly(torch.tensor([-np.inf, -1000.0, -126.0], device="cuda"), degree))
    assert np.all(tiny > 0) and np.all(tiny <= 2.0 ** -125)


# ---------------------------------------------------------------- back-to-back dependent calls

def test_back_to_back_calls_read_the_previous_output():
    # The forward and backward main kernels start launching while the kernel
    # before them finishes and wait for it before touching memory.  Chains of
    # small launch-bound calls where each reads the previous call's output
    # (O of one forward is Q of the next; the backward reads that forward's O
    # and L) must give what the oracle gives for the same chain.
    B, H, N, d, scale = 1, 2, 192, 64, 0.125
    q, k, v, do = inputs.draw_bf16(B, H, N, d, seed=31)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    x = qd
    for _ in range(6):
        o, lse = api.fa_fwd(x, kd, vd, True, scale)
        x = o
    dq, dk, dv = api.fa_bwd(x, kd, vd, *api.fa_fwd(x, kd, vd, True, scale), dod, True, scale)
    torch.cuda.synchronize()
    xr = q
    for _ in range(6):
        xr = torch.from_numpy(oracle.forward(xr, k, v, True, scale)[0]).to(torch.bfloat16)
    # each step's input is the GPU's previous bf16 output: compare the last
    # step against the oracle on that same input
    o_ref, l_ref = oracle.forward(x.cpu(), k, v, True, scale)
    o_last, l_last = api.fa_fwd(x, kd, vd, True, scale)
    torch.cuda.synchronize()
    assert max_abs(f64(o_last), o_ref) <= O_MAX_ABS
    assert max_abs(f64(l_last), l_ref) <= L_MAX_ABS
    # the chain itself stays close to the oracle's chain: each of its six
    # steps may add up to the O gate (bf16 rounding of its output)
    assert max_abs(f64(x), f64(xr)) <= 6 * O_MAX_ABS
    check_bwd(dq, dk, dv, x.cpu(), k, v, do, True, scale)
