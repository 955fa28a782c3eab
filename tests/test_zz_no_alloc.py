"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (for example a plugin inside another runtime that is handed only its
input and output tensors).  It takes its scratch from a fixed 32 MiB array in
the library instead of a caller workspace.

Checked here through the C ABI: two calls in a row (different inputs, so the
second would expose stale scratch) each match what fa_bwd with a caller
workspace produces, within the gradient tolerance every backward test uses,
for a small causal d = 128 case, a non-causal d = 64 case and a case whose
workspace is just under the array's 32 MiB (so the far end of the array is
used); a problem needing more than the array returns FA_ERR_WORKSPACE.  This
file is collected last on purpose."""
import ctypes
import math

import pytest
import torch

from exact_attention_76_gb300 import _lib, api, build, inputs
from tests.gpu_util import GRAD_REL_FRO, f64, rel_fro

pytestmark = pytest.mark.gpu

FA_ERR_WORKSPACE = 6


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("B,H,N,d,causal", [
    (2, 3, 333, 128, True),
    (1, 5, 700, 64, False),
    (1, 4, 16000, 128, True),   # workspace 33.02 MB, just under the 33.55 MB array
])
def test_noalloc_backward_matches_workspace_backward_twice(B, H, N, d, causal):
    build.build()
    lib = _lib.load()
    assert api.fa_bwd_workspace_size(B, H, N, d) <= 32 << 20
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((41, 42)):
        q, k, v, do = (t.cuda() for t in inputs.draw_bf16(B, H, N, d, seed))
        o, lse = api.fa_fwd(q, k, v, causal, scale)
        ref = api.fa_bwd(q, k, v, o, lse, do, causal, scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = lib.fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), _p(dq), _p(dk), _p(dv),
                                B, H, N, d, int(causal), scale, ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, f"call {call}: {_lib.STATUS_NAMES.get(st, st)}"
        torch.cuda.synchronize()
        for name, got, want in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
            e = rel_fro(f64(got), f64(want))
            assert e <= GRAD_REL_FRO, f"call {call}: {name} rel-Frobenius {e:.3e} against fa_bwd"
    assert api.fa_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = _lib.load()
    B, H, N, d = 4, 16, 8192, 128  # workspace ~ 269 MB > 32 MiB
    assert api.fa_bwd_workspace_size(B, H, N, d) > 32 << 20
    dummy = ctypes.c_void_p(0x10000)
    st = lib.fa_bwd_noalloc(*([dummy] * 9), B, H, N, d, 1, 0.088, None)
    assert st == FA_ERR_WORKSPACE
