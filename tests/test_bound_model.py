"""The tight per-element O bound the GPU parity tests apply
(tests/gpu_util.o_tight_bound), checked on the CPU against a model of the
kernel's arithmetic written here with numpy: S in fp32, p = exp(S - m) in fp32,
l summed from the unrounded p, P rounded to bf16 before P V, the sum in fp32,
O rounded to bf16.  The model must stay within the bound (its output rounding
alone can take an element close to it: half an ulp is the largest term), and
the same model with one extra key visible to each causal row (an off-by-one
mask) must fail it."""
import math

import numpy as np
import torch

import oracle
from exact_attention_76_gb300 import inputs
from tests.gpu_util import bf16_rne, o_tight_bound


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def _model_forward(q, k, v, causal, scale, extra_key=False):
    """One head, the kernel's roundings; extra_key lets row i also see key i+1."""
    q32, k32, v32 = (t.to(torch.float32).numpy() for t in (q, k, v))
    s = (q32 @ k32.T).astype(np.float32) * np.float32(scale)
    n = s.shape[0]
    if causal:
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        s = np.where(j > i + (1 if extra_key else 0), -np.inf, s).astype(np.float32)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m).astype(np.float32)
    ell = p.sum(axis=1, dtype=np.float32)
    o = (_bf16(p) @ v32).astype(np.float32) / ell[:, None]
    return _bf16(o)


def _case(N, d, causal, seed):
    q, k, v, _ = inputs.draw_bf16(1, 1, N, d, seed)
    scale = 1.0 / math.sqrt(d)
    o_ref, _ = oracle.forward(q, k, v, causal, scale)
    absv, _ = oracle.forward(q, k, v.abs(), causal, scale)
    return q[0, 0], k[0, 0], v[0, 0], o_ref[0, 0], absv[0, 0], scale


def test_model_of_the_kernel_arithmetic_is_within_the_bound():
    for N, d, causal, seed in ((300, 64, True, 1), (257, 128, False, 2), (64, 128, True, 3)):
        q, k, v, o_ref, absv, scale = _case(N, d, causal, seed)
        o = _model_forward(q, k, v, causal, scale)
        ratio = np.abs(o - o_ref) / o_tight_bound(o_ref, absv, N)
        assert ratio.max() <= 1.0, ratio.max()


def test_an_off_by_one_mask_breaks_the_bound():
    q, k, v, o_ref, absv, scale = _case(300, 64, True, 4)
    o = _model_forward(q, k, v, True, scale, extra_key=True)
    assert (np.abs(o - o_ref) > o_tight_bound(o_ref, absv, 300)).any()


def test_bf16_rne_rounds_to_nearest_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: even is 1
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5])
    assert np.array_equal(bf16_rne(x), [1.0, 1.0 + 2.0 ** -6, -2.5])
