"""Plain, slow, float64 CPU oracle for exact attention.  TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the bench's ``cpu_baseline`` /
``--impl reference`` legs may import this module.  It shares no code with the
CUDA path: it never imports the product package and the product never imports
it.  Everything here materialises the full N x N score and probability
matrices per (batch, head) and uses numpy float64; a matmul is the only library
primitive on the path.

Sources (page title, then the section or equation):
  * "FLASH-ATTN" (taking-lying-flat), FlashAttention-2 > Background: standard
    attention S = QK^T, P = softmax(S) row-wise, O = PV, parallel over batch
    and heads; and the backward chain dV = P^T dO, dP = dO V^T,
    dS = dsoftmax(dP), dQ = dS K, dK = dS^T Q.
  * "FLASH-ATTN", FlashAttention > Tiling and Recomputation: the (m, f, l)
    decomposition of softmax and the rule that merges two blocks' statistics.
  * "FLASH-ATTN", FlashAttention-2 > FlashAttention-2: the unscaled output
    accumulator O~ divided by diag(l) once after the loop, the saved statistic
    L = m + log(l), and the causal mask S_ij = -inf for j > i.
  * "FlashAttention 三代演进" (zoe.im), 第一代 > 洞察 2 Online Softmax: the running
    max / running sum recurrence over key tiles.

Readings where the pages are silent (each also listed in the design notes):
  * the pages write S = QK^T without a softmax scale; here S = scale * QK^T,
    applied before the mask and the softmax, and the chain rule through that
    product puts the same factor on dQ and dK;
  * L is in natural-log units of the scaled, masked logits: L = m + ln(l);
  * dsoftmax is the Jacobian of the row softmax: dS = P o (dP - D) with
    D_i = sum_j P_ij dP_ij;
  * causal attention is self-attention with N_q = N_k, so every row keeps j = i
    and no row is ever fully masked.
"""
from __future__ import annotations

import math

import numpy as np

LN2 = math.log(2.0)


def _f64(x) -> np.ndarray:
    """Upcast a numpy array or a CPU torch tensor of any float type to float64."""
    if hasattr(x, "detach"):  # a torch tensor (bf16, fp32, ...): exact upcast
        import torch
        x = x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Standard attention, one head: the definition written out.
# ---------------------------------------------------------------------------

def scores(q: np.ndarray, k: np.ndarray, causal: bool, scale: float) -> np.ndarray:
    """S = scale * Q K^T, with S_ij = -inf for j > i when causal.

    "FLASH-ATTN", FlashAttention-2 > Background (S = QK^T) and > FlashAttention-2
    (causal mask sets every S_ij with j > i to -inf).
    """
    s = scale * (q @ k.T)
    if causal:
        n_q, n_k = s.shape
        i = np.arange(n_q)[:, None]
        j = np.arange(n_k)[None, :]
        s = np.where(j > i, -np.inf, s)
    return s


def softmax_stats(s: np.ndarray):
    """Row statistics m(x) = max_i x_i, f(x) = exp(x - m(x)), l(x) = sum f(x).

    "FLASH-ATTN", FlashAttention > Tiling and Recomputation (definitions of m, f,
    l and softmax(x) = f(x) / l(x)).
    """
    m = s.max(axis=1)
    f = np.exp(s - m[:, None])
    ell = f.sum(axis=1)
    return m, f, ell


def head_forward(q, k, v, causal: bool, scale: float):
    """One (batch, head): returns O [N, d], L [N], P [N, N].

    O = softmax(S) V and L = m + ln(l) ("FLASH-ATTN", FlashAttention-2 >
    FlashAttention-2: LogSumExp statistic kept for the backward pass).
    """
    s = scores(q, k, causal, scale)
    m, f, ell = softmax_stats(s)
    p = f / ell[:, None]
    o = p @ v
    lse = m + np.log(ell)
    return o, lse, p


def head_backward(q, k, v, do, causal: bool, scale: float):
    """One (batch, head): returns dQ, dK, dV and D.

    "FLASH-ATTN", FlashAttention-2 > Background, the chain of five products:
    dV = P^T dO; dP = dO V^T; dS = dsoftmax(dP); dQ = dS K; dK = dS^T Q, with
    dsoftmax the row-softmax Jacobian dS = P o (dP - D), D_i = sum_j P_ij dP_ij,
    and the factor ``scale`` from S = scale * QK^T on dQ and dK.
    P is rebuilt here from the definition (no forward state is reused).
    """
    _, _, p = head_forward(q, k, v, causal, scale)
    dv = p.T @ do
    dp = do @ v.T
    dvec = (p * dp).sum(axis=1)
    ds = p * (dp - dvec[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, dvec


# ---------------------------------------------------------------------------
# Batched wrappers over [B, H, N, d].
# ---------------------------------------------------------------------------

def forward(q, k, v, causal: bool, scale: float, heads=None):
    """O [B,H,N,d] and L [B,H,N] in float64.  ``heads``: optional list of (b, h)
    to compute; other entries are left as NaN (used to sample large workloads)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    o = np.full((B, H, N, v.shape[-1]), np.nan)
    lse = np.full((B, H, N), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        ob, lb, _ = head_forward(q[b, h], k[b, h], v[b, h], causal, scale)
        o[b, h] = ob
        lse[b, h] = lb
    return o, lse


def backward(q, k, v, do, causal: bool, scale: float, heads=None):
    """dQ, dK, dV [B,H,N,d] in float64 (NaN outside ``heads`` when given)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        a, bb, c, _ = head_backward(q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
        dq[b, h], dk[b, h], dv[b, h] = a, bb, c
    return dq, dk, dv


def row_dot(o, do):
    """D_i = sum_k dO_ik O_ik per row, float64, over [B,H,N,d] -> [B,H,N].

    Equal to sum_j P_ij dP_ij (since O = PV and dP = dO V^T); the backward
    preprocess computes it this way because it needs only O and dO.
    """
    return (_f64(o) * _f64(do)).sum(axis=-1)


# ---------------------------------------------------------------------------
# The tiled one-pass algorithm, for the identity "online equals two-pass".
# ---------------------------------------------------------------------------

def online_softmax_vector(x: np.ndarray, block: int):
    """Page 1's one-pass softmax over one row: returns (softmax(x), m, l).

    "FlashAttention 三代演进", 第一代 > 洞察 2 Online Softmax: keep a running max and
    running sum; whenever a tile raises the max, multiply the old sum by
    exp(old_max - new_max).  The normalised vector is formed at the end from the
    final (m, l) ("FLASH-ATTN", Tiling and Recomputation: softmax = f / l).
    """
    x = np.asarray(x, dtype=np.float64)
    m = -np.inf
    ell = 0.0
    for start in range(0, x.size, block):
        t = x[start:start + block]
        m_new = max(m, float(t.max()))
        alpha = math.exp(m - m_new) if m != -np.inf else 0.0
        ell = ell * alpha + float(np.exp(t - m_new).sum())
        m = m_new
    return np.exp(x - m) / ell, m, ell


def head_forward_online(q, k, v, causal: bool, scale: float, block_c: int, tau: float = 0.0):
    """One head by the FlashAttention-2 recurrence over key blocks of ``block_c``.

    "FLASH-ATTN", FlashAttention-2 > FlashAttention-2: per key block j,
    m^(j) = max(m^(j-1), rowmax(S^(j))); O~^(j) = diag(e^{m^(j-1) - m^(j)}) O~^(j-1)
    + e^{S^(j) - m^(j)} V^(j); l likewise; after the last block O = diag(l)^-1 O~
    and L = m + log(l).  ``tau`` (natural-log units here) keeps the old max as the
    exponent's reference until the new block max exceeds it by more than tau;
    any tau >= 0 reaches the same O and L up to rounding.
    Fully masked key blocks (all j > i for the whole row block) are skipped, as
    the same section describes for causal attention.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n = q.shape[0]
    m_ref = np.full(n, -np.inf)
    ell = np.zeros(n)
    o_acc = np.zeros((n, v.shape[1]))
    for start in range(0, k.shape[0], block_c):
        if causal and start > n - 1:
            break
        kb = k[start:start + block_c]
        vb = v[start:start + block_c]
        s = scale * (q @ kb.T)
        if causal:
            i = np.arange(n)[:, None]
            j = start + np.arange(kb.shape[0])[None, :]
            s = np.where(j > i, -np.inf, s)
        blk_max = s.max(axis=1)
        raise_ref = blk_max > m_ref + tau
        m_new = np.where(raise_ref, blk_max, m_ref)
        with np.errstate(invalid="ignore"):
            alpha = np.where(np.isneginf(m_ref), 0.0, np.exp(m_ref - m_new))
        alpha = np.where(raise_ref, alpha, 1.0)
        with np.errstate(invalid="ignore"):
            e = np.exp(s - m_new[:, None])
        e = np.where(np.isneginf(s), 0.0, e)
        o_acc = alpha[:, None] * o_acc + e @ vb
        ell = alpha * ell + e.sum(axis=1)
        m_ref = m_new
    o = o_acc / ell[:, None]
    return o, m_ref + np.log(ell)


# ---------------------------------------------------------------------------
# FP8 forward reference.
# ---------------------------------------------------------------------------

def forward_fp8_reference(q_orig, k_orig, v_orig, causal: bool, scale: float, heads=None):
    """The FP8 forward's target: the same exact attention, in float64, on the
    inputs before quantisation ("FLASH-ATTN", Low-precision with FP8: per-tensor
    scaling keeps one scalar per tensor; the result it approximates is unchanged
    attention).  The gate therefore measures quantisation plus kernel error."""
    return forward(q_orig, k_orig, v_orig, causal, scale, heads=heads)


# ---------------------------------------------------------------------------
# FLOP convention used for throughput (not on the path).
# ---------------------------------------------------------------------------

def flops_forward(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """4 B H N^2 d (two N x N x d products), halved for causal by convention."""
    f = 4.0 * B * H * N * N * d
    return f / 2.0 if causal else f


def flops_backward(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """2.5 x the forward: five products against two."""
    return 2.5 * flops_forward(B, H, N, d, causal)


# ---------------------------------------------------------------------------
# FP8 storage with incoherent processing.
# ---------------------------------------------------------------------------

def hadamard_matrix(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (a power of two), scaled by 1/sqrt(d)
    so that it is orthogonal: H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]].

    "FLASH-ATTN", FlashAttention-3 > Low-precision with FP8 (incoherent
    processing multiplies Q and K by an orthogonal matrix M, which leaves
    (QM)(KM)^T = QK^T) and "FlashAttention 三代演进", 技术 4 (the matrix is a
    Hadamard transform).
    """
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    if h.shape[0] != d:
        raise ValueError("d must be a power of two")
    return h / math.sqrt(d)


def rotate_rows(x, d_axis_last=True):
    """x @ H for the last dimension (float64)."""
    x = _f64(x)
    return x @ hadamard_matrix(x.shape[-1])


def quantize_e4m3_reference(x):
    """Per-tensor e4m3 storage ("FLASH-ATTN", Low-precision with FP8: one scale
    per tensor): delta = amax|x| / 448 and code = e4m3_rne(x / delta).  The
    rounding is torch's float8_e4m3fn conversion (round to nearest even), applied
    to the float32 value of x / delta.  Returns (codes as uint8, delta)."""
    import torch
    x = _f64(x)
    amax = float(np.abs(x).max())
    delta = amax / 448.0 if amax > 0 else 1.0
    y = torch.from_numpy(np.clip(x / delta, -448.0, 448.0)).to(torch.float32)
    return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy(), delta


def dequantize_e4m3(codes, delta: float):
    """x ~= delta * e4m3(code), float64: the inverse of the per-tensor storage."""
    import torch
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return c * float(delta)


def quantize_e4m3_blocks_reference(x, block_rows: int):
    """Block e4m3 storage ("FLASH-ATTN", FlashAttention-3 > Low-precision with
    FP8, block quantisation: Q, K and V are cut into blocks of B_r x d or
    B_c x d rows and each block is quantised on its own, with one scale).

    x is [..., N, d]; every leading index is one sequence, and the blocks are
    rows [b*block_rows, (b+1)*block_rows) of a sequence (the last one may be
    shorter).  Per block: delta = amax|x| / 448 (1 for an all-zero block) and
    code = e4m3_rne(x / delta), the rounding being torch's float8_e4m3fn
    conversion of the float32 value of x / delta.  Returns (codes as uint8 with
    the shape of x, deltas [..., ceil(N / block_rows)] float64)."""
    import torch
    x = _f64(x)
    N = x.shape[-2]
    nb = -(-N // block_rows)
    codes = np.empty(x.shape, dtype=np.uint8)
    deltas = np.empty(x.shape[:-2] + (nb,), dtype=np.float64)
    for b in range(nb):
        rows = slice(b * block_rows, min(N, (b + 1) * block_rows))
        blk = x[..., rows, :]
        amax = np.abs(blk).max(axis=(-2, -1))
        delta = np.where(amax > 0, amax / 448.0, 1.0)
        y = np.clip(blk / delta[..., None, None], -448.0, 448.0)
        codes[..., rows, :] = torch.from_numpy(y).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        deltas[..., b] = delta
    return codes, deltas


def dequantize_e4m3_blocks(codes, deltas, block_rows: int):
    """x ~= delta_block * e4m3(code): the inverse mapping of the block storage
    above (float64)."""
    import torch
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scale = np.repeat(_f64(deltas), block_rows, axis=-1)[..., : c.shape[-2]]
    return c * scale[..., None]


# ---------------------------------------------------------------------------
# Causal sliding window.
# ---------------------------------------------------------------------------

def _window_bias(n: int, window: int) -> np.ndarray:
    """0 where query i sees key j (i - window < j <= i), -inf elsewhere.
    "FLASH-ATTN" names sliding window among the supported mask variants; the
    pages give no definition, this is the reading taken (the `window` most
    recent keys, the query's own included)."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return np.where((j <= i) & (j > i - window), 0.0, -np.inf)


def forward_window(q, k, v, window: int, scale: float):
    """O [B,H,N,d], L [B,H,N] (float64) of causal sliding-window attention:
    the definition S = scale Q K^T + mask, P = softmax(S), O = P V,
    L = m + ln l, with the window mask above; k and v may have fewer heads
    (grouped queries, head h reads h // (H // Hkv))."""
    q, k, v = _f64(q), _expand_kv(k, _f64(q).shape[1]), _expand_kv(v, _f64(q).shape[1])
    B, H, N, _ = q.shape
    bias = _window_bias(N, window)
    o = np.empty(q.shape[:3] + (v.shape[-1],))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h] @ k[b, h].T) + bias
            m, f, ell = softmax_stats(s)
            o[b, h] = (f / ell[:, None]) @ v[b, h]
            lse[b, h] = m + np.log(ell)
    return o, lse


def backward_window(q, k, v, do, window: int, scale: float):
    """dQ [B,H,N,d] and dK, dV [B,Hkv,N,d] (float64) of forward_window: the
    five products of the backward with P from the windowed softmax; dK and dV
    of a shared key/value head are summed over its query heads."""
    H = _f64(q).shape[1]
    Hkv = _f64(k).shape[1]
    q, do = _f64(q), _f64(do)
    kx, vx = _expand_kv(k, H), _expand_kv(v, H)
    B, _, N, _ = q.shape
    bias = _window_bias(N, window)
    dq = np.empty_like(q)
    dkx = np.empty_like(kx)
    dvx = np.empty_like(vx)
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h] @ kx[b, h].T) + bias
            m, f, ell = softmax_stats(s)
            p = f / ell[:, None]
            dvx[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ vx[b, h].T
            ds = p * (dp - (p * dp).sum(axis=1)[:, None])
            dq[b, h] = scale * (ds @ kx[b, h])
            dkx[b, h] = scale * (ds.T @ q[b, h])
    g = H // Hkv
    dk = dkx.reshape(B, Hkv, g, N, -1).sum(axis=2)
    dv = dvx.reshape(B, Hkv, g, N, -1).sum(axis=2)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Decode: one query row against a key/value cache.
# ---------------------------------------------------------------------------

def decode(q, k, v, scale: float):
    """q [B, H, d], k and v [B, Hkv, N, d] -> O [B, H, d], L [B, H] (float64).

    One query row per (batch, head) attending to every key of the cache, no
    mask: standard attention ("FLASH-ATTN", FlashAttention-2 > Background) with
    a single query, the decode case of "FlashAttention 三代演进".  Query head h
    reads key/value head h // (H // Hkv)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, d = q.shape
    g = H // k.shape[1]
    o = np.empty((B, H, v.shape[-1]))
    lse = np.empty((B, H))
    for b in range(B):
        for h in range(H):
            ob, lb, _ = head_forward(q[b, h][None, :], k[b, h // g], v[b, h // g], False, scale)
            o[b, h] = ob[0]
            lse[b, h] = lb[0]
    return o, lse


# ---------------------------------------------------------------------------
# Grouped-query attention.
# ---------------------------------------------------------------------------

def _expand_kv(x, H):
    """[B, Hkv, N, d] -> [B, H, N, d]: query head h reads key/value head
    h // (H // Hkv) ("FLASH-ATTN", FlashAttention-2 > FlashAttention-2: the
    shared heads are addressed by index, not copied; copying here is the plain
    definition)."""
    x = _f64(x)
    return np.repeat(x, H // x.shape[1], axis=1)


def forward_gqa(q, k, v, causal: bool, scale: float, heads=None):
    """Grouped-query forward: standard attention with each query head reading
    its group's key and value head."""
    H = _f64(q).shape[1]
    return forward(q, _expand_kv(k, H), _expand_kv(v, H), causal, scale, heads=heads)


def backward_gqa(q, k, v, do, causal: bool, scale: float):
    """Grouped-query backward: per query head as in `backward`, then dK and dV
    of a shared head summed over the query heads that read it (same section)."""
    H = _f64(q).shape[1]
    Hkv = _f64(k).shape[1]
    dq, dk, dv = backward(q, _expand_kv(k, H), _expand_kv(v, H), do, causal, scale)
    B, _, N, d = dk.shape
    g = H // Hkv
    return dq, dk.reshape(B, Hkv, g, N, d).sum(axis=2), dv.reshape(B, Hkv, g, N, d).sum(axis=2)
