"""Python face of the C ABI (include/fa.h), one function per entry point and
with the same names.  PyTorch supplies device memory and the stream; every
step of the computation runs in the library's CUDA kernels.

Tensors are CUDA, contiguous, [B, H, N, d]; bf16 unless stated; statistics
([B, H, N]) are fp32.  Outputs may be passed in (pre-allocated) or are
allocated here with torch.
"""
from __future__ import annotations

import torch

from . import _lib


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor):
    return t.data_ptr()


def _check(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def fa_fwd(q, k, v, causal: bool, scale: float, o=None, lse=None, stream=None):
    """O = softmax(scale QK^T [+ causal mask]) V and L = logsumexp of the scaled logits."""
    lib = _lib.load()
    B, H, N, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, (B, H, N, d))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check(o, "o", torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    _lib.check("fa_fwd", lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(bool(causal)),
                                    float(scale), _stream_ptr(stream)))
    return o, lse


def fa_fwd_gqa(q, k, v, causal: bool, scale: float, o=None, lse=None, stream=None):
    """Grouped-query forward: q [B,H,N,d], k and v [B,Hkv,N,d] with Hkv dividing H."""
    lib = _lib.load()
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    _check(q, "q", torch.bfloat16, (B, H, N, d))
    for t, n in ((k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, (B, Hkv, N, d))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "o", torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    _lib.check("fa_fwd_gqa", lib.fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                            int(bool(causal)), float(scale), _stream_ptr(stream)))
    return o, lse


def fa_bwd_gqa(q, k, v, o, lse, dO, causal: bool, scale: float, dq=None, dk=None, dv=None, workspace=None,
               stream=None):
    """Grouped-query backward; dk and dv have k's and v's shape [B,Hkv,N,d]."""
    lib = _lib.load()
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    for t, n in ((q, "q"), (o, "o"), (dO, "dO")):
        _check(t, n, torch.bfloat16, (B, H, N, d))
    for t, n in ((k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, (B, Hkv, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_gqa_workspace_size(B, H, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _lib.check("fa_bwd_gqa", lib.fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                            _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, H, Hkv, N, d,
                                            int(bool(causal)), float(scale), _stream_ptr(stream)))
    return dq, dk, dv


def fa_fwd_window(q, k, v, window: int, scale: float, o=None, lse=None, stream=None):
    """Causal attention where query i sees keys i-window+1 .. i; q [B,H,N,d],
    k and v [B,Hkv,N,d]."""
    lib = _lib.load()
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    _check(q, "q", torch.bfloat16, (B, H, N, d))
    for t, n in ((k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, (B, Hkv, N, d))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "o", torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    _lib.check("fa_fwd_window", lib.fa_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                                  int(window), float(scale), _stream_ptr(stream)))
    return o, lse


def fa_bwd_window(q, k, v, o, lse, dO, window: int, scale: float, dq=None, dk=None, dv=None, workspace=None,
                  stream=None):
    """Backward of fa_fwd_window; dk and dv have k's and v's shape."""
    lib = _lib.load()
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    for t, n in ((q, "q"), (o, "o"), (dO, "dO")):
        _check(t, n, torch.bfloat16, (B, H, N, d))
    for t, n in ((k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, (B, Hkv, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=q.device)
    _lib.check("fa_bwd_window", lib.fa_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                                  _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, H, Hkv,
                                                  N, d, int(window), float(scale), _stream_ptr(stream)))
    return dq, dk, dv


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(_lib.load().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd_gqa_workspace_size(B: int, H: int, Hkv: int, N: int, d: int) -> int:
    """Workspace bytes for fa_bwd_gqa (room for the dK and dV accumulators when
    it would split a group's query heads over CTAs)."""
    return int(_lib.load().fa_bwd_gqa_workspace_size(B, H, Hkv, N, d))


def fa_bwd(q, k, v, o, lse, dO, causal: bool, scale: float, dq=None, dk=None, dv=None, workspace=None,
           stream=None):
    """dQ, dK, dV of O = softmax(scale QK^T [+mask]) V for upstream gradient dO."""
    lib = _lib.load()
    B, H, N, d = q.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO")):
        _check(t, n, torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, torch.bfloat16, (B, H, N, d))
    need = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    _lib.check("fa_bwd", lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                    _ptr(dv), _ptr(workspace), workspace.numel(), B, H, N, d, int(bool(causal)),
                                    float(scale), _stream_ptr(stream)))
    return dq, dk, dv


def fa_bwd_preprocess(o, dO, D=None, dq_acc=None, stream=None):
    """D = rowsum(dO * O) in fp32 and a zeroed fp32 dQ accumulator."""
    lib = _lib.load()
    B, H, N, d = o.shape
    _check(o, "o", torch.bfloat16)
    _check(dO, "dO", torch.bfloat16, (B, H, N, d))
    D = torch.empty((B, H, N), dtype=torch.float32, device=o.device) if D is None else D
    dq_acc = torch.empty((B, H, N, d), dtype=torch.float32, device=o.device) if dq_acc is None else dq_acc
    _check(D, "D", torch.float32, (B, H, N))
    _check(dq_acc, "dq_acc", torch.float32, (B, H, N, d))
    _lib.check("fa_bwd_preprocess", lib.fa_bwd_preprocess(_ptr(o), _ptr(dO), _ptr(D), _ptr(dq_acc), B, H, N, d,
                                                          _stream_ptr(stream)))
    return D, dq_acc


def fa_bwd_main(q, k, v, lse, dO, D, dq_acc, causal: bool, scale: float, dk=None, dv=None, stream=None):
    """dK, dV (bf16) and dS K added into dq_acc (fp32)."""
    lib = _lib.load()
    B, H, N, d = q.shape
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _lib.check("fa_bwd_main", lib.fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(dO), _ptr(D),
                                              _ptr(dq_acc), _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)),
                                              float(scale), _stream_ptr(stream)))
    return dk, dv


def fa_bwd_dq_convert(dq_acc, scale: float, dq=None, stream=None):
    """dQ = bf16(scale * dq_acc)."""
    lib = _lib.load()
    B, H, N, d = dq_acc.shape
    _check(dq_acc, "dq_acc", torch.float32)
    dq = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dq_acc.device) if dq is None else dq
    _lib.check("fa_bwd_dq_convert", lib.fa_bwd_dq_convert(_ptr(dq_acc), _ptr(dq), B, H, N, d, float(scale),
                                                          _stream_ptr(stream)))
    return dq


def fa_fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, causal: bool, scale: float, o=None, lse=None,
               stream=None):
    """FP8 forward: q8/k8/v8 are e4m3 codes (torch.uint8 or float8_e4m3fn), descales are
    1-element fp32 CUDA tensors; returns bf16 O and fp32 L."""
    lib = _lib.load()
    B, H, N, d = q8.shape
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError(f"{n}: expected e4m3 codes")
        _check(t, n, t.dtype, (B, H, N, d))
    for t, n in ((descale_q, "descale_q"), (descale_k, "descale_k"), (descale_v, "descale_v")):
        _check(t, n, torch.float32)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _lib.check("fa_fwd_fp8", lib.fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(descale_q), _ptr(descale_k),
                                            _ptr(descale_v), _ptr(o), _ptr(lse), B, H, N, d, int(bool(causal)),
                                            float(scale), _stream_ptr(stream)))
    return o, lse


def fa_fp8_quantize(x, hadamard: bool, codes=None, descale=None, stream=None):
    """Per-tensor e4m3 codes of x (optionally rotated by the normalised Hadamard
    transform along the last dimension) and the fp32 descale.  x: CUDA fp32 or
    bf16, last dimension 64 or 128.  Returns (codes uint8 of x's shape, descale
    as a 1-element fp32 tensor)."""
    lib = _lib.load()
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x: expected fp32 or bf16")
    _check(x, "x", x.dtype)
    d = x.shape[-1]
    rows = x.numel() // d
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if codes is None else codes
    descale = torch.empty(1, dtype=torch.float32, device=x.device) if descale is None else descale
    _check(codes, "codes", torch.uint8, tuple(x.shape))
    _check(descale, "descale", torch.float32)
    _lib.check("fa_fp8_quantize", lib.fa_fp8_quantize(_ptr(x), 1 if x.dtype == torch.bfloat16 else 0,
                                                      int(bool(hadamard)), _ptr(codes), _ptr(descale), rows, d,
                                                      _stream_ptr(stream)))
    return codes, descale


FP8_BLOCK_Q = 128   # rows of Q per scale (FA_FP8_BLOCK_Q)
FP8_BLOCK_KV = 64   # rows of K and of V per scale (FA_FP8_BLOCK_KV)


def fa_fwd_fp8_blocks(q8, k8, v8, descale_q, descale_k, descale_v, causal: bool, scale: float, o=None, lse=None,
                      stream=None):
    """FP8 forward on block-quantised inputs: descale_q is [B*H, ceil(N/128)],
    descale_k and descale_v are [B*H, ceil(N/64)] fp32 CUDA tensors (one scale
    per block of rows).  Returns bf16 O and fp32 L."""
    lib = _lib.load()
    B, H, N, d = q8.shape
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError(f"{n}: expected e4m3 codes")
        _check(t, n, t.dtype, (B, H, N, d))
    nq, nk = -(-N // FP8_BLOCK_Q), -(-N // FP8_BLOCK_KV)
    _check(descale_q, "descale_q", torch.float32, (B * H, nq))
    _check(descale_k, "descale_k", torch.float32, (B * H, nk))
    _check(descale_v, "descale_v", torch.float32, (B * H, nk))
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _lib.check("fa_fwd_fp8_blocks", lib.fa_fwd_fp8_blocks(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(descale_q),
                                                          _ptr(descale_k), _ptr(descale_v), _ptr(o), _ptr(lse), B, H,
                                                          N, d, int(bool(causal)), float(scale),
                                                          _stream_ptr(stream)))
    return o, lse


def fa_fp8_quantize_blocks(x, hadamard: bool, block_rows: int, codes=None, descale=None, stream=None):
    """Block e4m3 codes of x [..., N, d] (every leading index one sequence),
    one scale per block_rows rows of a sequence, optionally after the
    normalised Hadamard rotation of each row.  Returns (codes uint8 of x's
    shape, descale fp32 [prod(leading dims), ceil(N / block_rows)])."""
    lib = _lib.load()
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x: expected fp32 or bf16")
    _check(x, "x", x.dtype)
    N, d = x.shape[-2], x.shape[-1]
    seqs = x.numel() // (N * d)
    nb = -(-N // int(block_rows))
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if codes is None else codes
    descale = torch.empty((seqs, nb), dtype=torch.float32, device=x.device) if descale is None else descale
    _check(codes, "codes", torch.uint8, tuple(x.shape))
    _check(descale, "descale", torch.float32, (seqs, nb))
    _lib.check("fa_fp8_quantize_blocks", lib.fa_fp8_quantize_blocks(
        _ptr(x), 1 if x.dtype == torch.bfloat16 else 0, int(bool(hadamard)), int(block_rows), _ptr(codes),
        _ptr(descale), seqs, N, d, _stream_ptr(stream)))
    return codes, descale


def fa_decode_workspace_size(B: int, H: int, Hkv: int, N: int, d: int) -> int:
    return int(_lib.load().fa_decode_workspace_size(B, H, Hkv, N, d))


def fa_decode(q, k, v, scale: float, o=None, lse=None, workspace=None, stream=None):
    """One query row per (batch, head) against the key/value cache k, v
    [B, Hkv, N, d]; q is [B, H, d] bf16.  Returns bf16 O [B, H, d] and fp32 L
    [B, H]."""
    lib = _lib.load()
    B, H, d = q.shape
    _, Hkv, N, _ = k.shape
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (B, Hkv, N, d))
    _check(v, "v", torch.bfloat16, (B, Hkv, N, d))
    o = torch.empty((B, H, d), dtype=torch.bfloat16, device=q.device) if o is None else o
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "o", torch.bfloat16, (B, H, d))
    _check(lse, "lse", torch.float32, (B, H))
    ws_bytes = fa_decode_workspace_size(B, H, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    _lib.check("fa_decode", lib.fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                          workspace.numel(), B, H, Hkv, N, d, float(scale), _stream_ptr(stream)))
    return o, lse


def fa_measure_ex2_rate(stream=None) -> float:
    """exp2 results per clock per SM of the special-function unit (a measurement;
    synchronises the stream).  Its scratch is allocated here with torch."""
    import ctypes
    lib = _lib.load()
    nbytes = int(lib.fa_measure_ex2_rate_scratch_size())
    if nbytes == 0:
        raise RuntimeError("fa_measure_ex2_rate_scratch_size: no current CUDA device")
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = ctypes.c_float(0.0)
    _lib.check("fa_measure_ex2_rate", lib.fa_measure_ex2_rate(ctypes.byref(out), _ptr(scratch), nbytes,
                                                               _stream_ptr(stream)))
    return float(out.value)


def fa_debug_exp2_poly(x, degree: int, y=None, stream=None):
    """2^x by the library's FMA-pipe polynomial (test hook); x fp32 CUDA."""
    lib = _lib.load()
    _check(x, "x", torch.float32)
    y = torch.empty_like(x) if y is None else y
    _check(y, "y", torch.float32, tuple(x.shape))
    _lib.check("fa_debug_exp2_poly", lib.fa_debug_exp2_poly(_ptr(x), _ptr(y), x.numel(), int(degree),
                                                             _stream_ptr(stream)))
    return y


def fa_status_string(status: int) -> str:
    return _lib.load().fa_status_string(int(status)).decode()


def fa_device_error(stream=None) -> int:
    """Synchronises the stream; returns the status code (0 = FA_OK, 5 = FA_ERR_TIMEOUT)."""
    return int(_lib.load().fa_device_error(_stream_ptr(stream)))


def fa_debug_wait_timeout(limit_us: int, stream=None) -> int:
    return int(_lib.load().fa_debug_wait_timeout(int(limit_us), _stream_ptr(stream)))
