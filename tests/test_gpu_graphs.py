"""The compute entry points inside CUDA graphs.

Each case captures a call sequence on a side stream, replays the graph on new
inputs copied into the captured buffers, and compares the results with the
same calls made eagerly:
- a forward + backward step;
- a grouped decode;
- FP8 storage followed by the FP8 forward.

The calls only enqueue asynchronous work on their stream: kernels, programmatic
dependent launches and memsets. That is what lets a capture hold them. Results
are bit-identical except dQ, whose fp32 partial sums from different key blocks
are added in the order the CTAs finish."""
import math

import pytest
import torch

from exact_attention_76_gb300 import api, inputs
from tests.gpu_util import f64, rel_fro

pytestmark = pytest.mark.gpu


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # first calls outside the capture (module loading, function attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_forward_backward_step_in_a_graph(d, causal):
    B, H, N = 2, 3, 333
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (t.cuda() for t in inputs.draw_bf16(B, H, N, d, 51))
    o, lse = torch.empty_like(q), torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(api.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")

    def step():
        api.fa_fwd(q, k, v, causal, scale, o=o, lse=lse)
        api.fa_bwd(q, k, v, o, lse, do, causal, scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    g = _capture(step)
    for seed in (52, 53):
        new = [t.cuda() for t in inputs.draw_bf16(B, H, N, d, seed)]
        for dst, src in zip((q, k, v, do), new):
            dst.copy_(src)
        g.replay()
        ref_o, ref_lse = api.fa_fwd(*new[:3], causal, scale)
        ref_dq, ref_dk, ref_dv = api.fa_bwd(*new[:3], ref_o, ref_lse, new[3], causal, scale)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
        assert torch.equal(dk, ref_dk) and torch.equal(dv, ref_dv)
        assert rel_fro(f64(dq), f64(ref_dq)) <= 1e-3
    assert api.fa_device_error() == 0


def test_grouped_decode_in_a_graph():
    B, H, Hkv, N, d = 3, 8, 2, 3000, 128
    scale = 1.0 / math.sqrt(d)
    gen = torch.Generator(device="cuda").manual_seed(7)

    def draw():
        return (torch.randn(B, H, d, device="cuda", generator=gen).to(torch.bfloat16),
                torch.randn(B, Hkv, N, d, device="cuda", generator=gen).to(torch.bfloat16),
                torch.randn(B, Hkv, N, d, device="cuda", generator=gen).to(torch.bfloat16))

    q, k, v = draw()
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, dtype=torch.float32, device="cuda")
    ws = torch.empty(api.fa_decode_workspace_size(B, H, Hkv, N, d), dtype=torch.uint8, device="cuda")
    g = _capture(lambda: api.fa_decode(q, k, v, scale, o=o, lse=lse, workspace=ws))
    for _ in range(2):
        new = draw()
        for dst, src in zip((q, k, v), new):
            dst.copy_(src)
        g.replay()
        ref_o, ref_lse = api.fa_decode(*new, scale)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert api.fa_device_error() == 0


def test_fp8_storage_and_forward_in_a_graph():
    B, H, N, d, causal = 1, 2, 500, 128, True
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.cuda() for t in inputs.draw_outlier_fp32(B, H, N, d, seed=61))
    codes = [torch.empty(q.shape, dtype=torch.uint8, device="cuda") for _ in range(3)]
    desc = [torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3)]
    o, lse = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda"), torch.empty(B, H, N, device="cuda")

    def run():
        for t, rot, c, s in zip((q, k, v), (True, True, False), codes, desc):
            api.fa_fp8_quantize(t, rot, codes=c, descale=s)
        api.fa_fwd_fp8(*codes, *desc, causal, scale, o=o, lse=lse)

    g = _capture(run)
    for seed in (62, 63):
        new = [t.cuda() for t in inputs.draw_outlier_fp32(B, H, N, d, seed=seed)]
        for dst, src in zip((q, k, v), new):
            dst.copy_(src)
        g.replay()
        ref = [api.fa_fp8_quantize(t, rot) for t, rot in zip(new, (True, True, False))]
        ref_o, ref_lse = api.fa_fwd_fp8(*[c for c, _ in ref], *[s for _, s in ref], causal, scale)
        torch.cuda.synchronize()
        for (rc, rs), c, s in zip(ref, codes, desc):
            assert torch.equal(c, rc) and torch.equal(s, rs)
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert api.fa_device_error() == 0
