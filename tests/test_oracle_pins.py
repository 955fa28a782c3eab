"""Pins for the float64 oracle: each check comes from something other than the
oracle's own formula -- closed forms, invariants, the pages' identities, brute
force on tiny inputs, finite differences, or a library routine.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_76_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def rand_qkv(n, d, seed, n_k=None):
    r = rng(seed)
    n_k = n if n_k is None else n_k
    return r.standard_normal((n, d)), r.standard_normal((n_k, d)), r.standard_normal((n_k, d))


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_values(causal):
    # Q = 0 makes every score 0: P is uniform over the unmasked keys.
    n, d = 37, 5
    _, k, v = rand_qkv(n, d, 1)
    q = np.zeros((n, d))
    o, lse, _ = oracle.head_forward(q, k, v, causal, 0.3)
    for i in range(n):
        cnt = i + 1 if causal else n
        np.testing.assert_allclose(o[i], v[:cnt].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(lse[i] - math.log(cnt)) < 1e-13


def test_causal_row_zero_is_first_value():
    n, d, s = 19, 8, 0.7
    q, k, v = rand_qkv(n, d, 2)
    o, lse, _ = oracle.head_forward(q, k, v, True, s)
    np.testing.assert_array_equal(o[0], v[0])
    assert abs(lse[0] - s * float(q[0] @ k[0])) < 1e-13


def test_dominant_logit_selects_its_value_row():
    n, d, s = 16, 8, 1.0
    q, k, v = rand_qkv(n, d, 3)
    i, jstar, c = 5, 11, 60.0
    k = k * 0.01
    k[jstar] = c * q[i] / np.linalg.norm(q[i])
    o, _, _ = oracle.head_forward(q, k, v, False, s)
    # every other logit is at most |q_i| * max|k_j| with k_j tiny
    gap = s * c * np.linalg.norm(q[i]) - s * np.linalg.norm(q[i]) * np.abs(k[np.arange(n) != jstar]).sum(1).max()
    bound = (n - 1) * math.exp(-gap) * 2 * np.abs(v).max()
    assert np.abs(o[i] - v[jstar]).max() <= bound + 1e-15


def test_two_key_softmax_is_logistic():
    # With two keys the softmax weight of key 0 is the logistic function of the
    # score difference: sigma(x) = 1 / (1 + e^-x).
    q = np.array([[1.5, -0.5]])
    k = np.array([[0.8, 0.3], [-0.2, 0.9]])
    v = np.array([[2.0, -1.0], [0.5, 4.0]])
    s = 0.9
    x = s * (q[0] @ k[0] - q[0] @ k[1])
    w0 = 1.0 / (1.0 + math.exp(-x))
    o, lse, _ = oracle.head_forward(q, k, v, False, s)
    np.testing.assert_allclose(o[0], w0 * v[0] + (1 - w0) * v[1], rtol=0, atol=1e-15)
    s0, s1 = s * q[0] @ k[0], s * q[0] @ k[1]
    assert abs(lse[0] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-14


# ---------------------------------------------------------------- brute force

def brute_force_head(q, k, v, causal, s):
    """Scalar loops with math.exp: independent of the vectorised oracle."""
    n, d = len(q), len(q[0])
    o, lse = [], []
    for i in range(n):
        keys = range(i + 1) if causal else range(len(k))
        logits = [s * sum(q[i][t] * k[j][t] for t in range(d)) for j in keys]
        mx = max(logits)
        w = [math.exp(x - mx) for x in logits]
        tot = sum(w)
        o.append([sum(w[a] * v[j][t] for a, j in enumerate(keys)) / tot for t in range(len(v[0]))])
        lse.append(mx + math.log(tot))
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(causal):
    q, k, v = rand_qkv(6, 3, 4)
    o, lse, _ = oracle.head_forward(q, k, v, causal, 0.45)
    ob, lb = brute_force_head(q.tolist(), k.tolist(), v.tolist(), causal, 0.45)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-14)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    q, k, v = rand_qkv(50, 16, 5)
    _, _, p = oracle.head_forward(q, k, v, causal, 0.25)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    if causal:
        assert np.all(p[np.triu_indices(50, 1)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_shift_of_keys(causal):
    # K_j <- K_j + c for all j adds s*q_i.c to every logit of row i: O is
    # unchanged and L_i moves by exactly that amount.
    n, d, s = 40, 6, 0.4
    q, k, v = rand_qkv(n, d, 6)
    c = rng(7).standard_normal(d)
    o1, l1, _ = oracle.head_forward(q, k, v, causal, s)
    o2, l2, _ = oracle.head_forward(q, k + c, v, causal, s)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + s * (q @ c), rtol=0, atol=1e-12)


def test_key_value_permutation_non_causal():
    q, k, v = rand_qkv(33, 7, 8)
    perm = rng(9).permutation(33)
    o1, l1, _ = oracle.head_forward(q, k, v, False, 0.5)
    o2, l2, _ = oracle.head_forward(q, k[perm], v[perm], False, 0.5)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_orthogonal_rotation_of_q_and_k(causal):
    # "FLASH-ATTN", Low-precision with FP8 (incoherent processing): for an
    # orthogonal M, (QM)(KM)^T = QK^T, so the output does not change.
    n, d = 30, 16
    q, k, v = rand_qkv(n, d, 10)
    m, _ = np.linalg.qr(rng(11).standard_normal((d, d)))
    o1, l1, _ = oracle.head_forward(q, k, v, causal, 0.25)
    o2, l2, _ = oracle.head_forward(q @ m, k @ m, v, causal, 0.25)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_column_sums(causal):
    # Rows of dS sum to zero, so sum_j dK_j = 0; rows of P sum to one, so
    # sum_j dV_j = sum_i dO_i.
    n, d = 45, 8
    q, k, v = rand_qkv(n, d, 12)
    do = rng(13).standard_normal((n, d))
    dq, dk, dv, dvec = oracle.head_backward(q, k, v, do, causal, 0.35)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), rtol=0, atol=1e-12)
    o, _, _ = oracle.head_forward(q, k, v, causal, 0.35)
    np.testing.assert_allclose(dvec, (do * o).sum(axis=1), rtol=0, atol=1e-12)


def test_row_dot_matches_definition():
    q, k, v = rand_qkv(20, 4, 14)
    do = rng(15).standard_normal((20, 4))
    o, _, p = oracle.head_forward(q, k, v, True, 0.5)
    dp = do @ v.T
    got = oracle.row_dot(o[None, None], do[None, None])[0, 0]
    np.testing.assert_allclose(got, (p * dp).sum(1), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- online == two-pass

@pytest.mark.parametrize("block", [1, 7, 64, 200])
def test_online_softmax_vector(block):
    x = rng(16).standard_normal(200) * 5
    y, m, ell = oracle.online_softmax_vector(x, block)
    e = np.exp(x - x.max())
    np.testing.assert_allclose(y, e / e.sum(), rtol=0, atol=1e-15)
    assert m == x.max()
    assert abs(ell - e.sum()) < 1e-12 * e.sum()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 7, 64, 130])
@pytest.mark.parametrize("tau", [0.0, 8 * math.log(2.0)])
def test_online_fa2_equals_definition(causal, block, tau):
    n, d, s = 130, 16, 0.3
    q, k, v = rand_qkv(n, d, 17)
    q *= 3.0  # spread the logits so the running max moves between blocks
    o1, l1, _ = oracle.head_forward(q, k, v, causal, s)
    o2, l2 = oracle.head_forward_online(q, k, v, causal, s, block, tau)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("causal", [False, True])
def test_gradients_by_central_differences(causal):
    n, d, s, h = 8, 4, 0.6, 1e-6
    q, k, v = rand_qkv(n, d, 18)
    do = rng(19).standard_normal((n, d))

    def loss(qq, kk, vv):
        o, _, _ = oracle.head_forward(qq, kk, vv, causal, s)
        return float((o * do).sum())

    dq, dk, dv, _ = oracle.head_backward(q, k, v, do, causal, s)
    for x, g, idx in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        fd = np.zeros_like(x)
        for a in range(n):
            for b in range(d):
                xp = x.copy(); xp[a, b] += h
                xm = x.copy(); xm[a, b] -= h
                args_p = [q, k, v]; args_p[idx] = xp
                args_m = [q, k, v]; args_m[idx] = xm
                fd[a, b] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(fd - g).max() / np.abs(g).max()
        assert err <= 1e-6, (idx, err)


def test_gradients_fd_on_tiny_workload_entries():
    w = inputs.TINY
    q, k, v, do = (t.double().numpy() for t in inputs.draw_fp32(w.B, w.H, w.N, w.d, w.seed))
    b, hh = 0, 1
    qh, kh, vh, doh = q[b, hh], k[b, hh], v[b, hh], do[b, hh]
    dq, dk, dv, _ = oracle.head_backward(qh, kh, vh, doh, w.causal, w.scale)
    h = 1e-6

    def loss(qq, kk, vv):
        o, _, _ = oracle.head_forward(qq, kk, vv, w.causal, w.scale)
        return float((o * doh).sum())

    for (idx, g) in ((0, dq), (1, dk), (2, dv)):
        for (a, c) in ((0, 0), (17, 33), (127, 63)):
            base = [qh, kh, vh]
            xp = [t.copy() for t in base]; xp[idx][a, c] += h
            xm = [t.copy() for t in base]; xm[idx][a, c] -= h
            fd = (loss(*xp) - loss(*xm)) / (2 * h)
            assert abs(fd - g[a, c]) <= 1e-6 * max(1.0, np.abs(g).max()), (idx, a, c, fd, g[a, c])


# ---------------------------------------------------------------- library routine

@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_sdpa_float64(causal):
    w = inputs.GPT2
    q, k, v, do = inputs.draw_bf16(1, 3, 256, w.d, w.seed)
    q64, k64, v64, do64 = (t.double().requires_grad_(True) for t in (q, k, v, do))
    o_t = torch.nn.functional.scaled_dot_product_attention(q64, k64, v64, is_causal=causal, scale=w.scale)
    o_t.backward(do64)
    o, lse = oracle.forward(q, k, v, causal, w.scale)
    np.testing.assert_allclose(o, o_t.detach().numpy(), rtol=0, atol=1e-12)
    s = w.scale * (q64.detach() @ k64.detach().transpose(-1, -2))
    if causal:
        s = s.masked_fill(torch.ones(256, 256, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)
    dq, dk, dv = oracle.backward(q, k, v, do, causal, w.scale)
    np.testing.assert_allclose(dq, q64.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, k64.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, v64.grad.numpy(), rtol=0, atol=1e-11)


def test_sampled_heads_match_full():
    q, k, v, do = inputs.draw_bf16(2, 3, 64, 16, 5)
    o_full, l_full = oracle.forward(q, k, v, True, 0.25)
    o_s, l_s = oracle.forward(q, k, v, True, 0.25, heads=[(1, 2)])
    np.testing.assert_array_equal(o_s[1, 2], o_full[1, 2])
    assert np.isnan(o_s[0, 0]).all() and np.isnan(l_s[0, 1]).all()


# ---------------------------------------------------------------- page figures

def test_page_figures():
    items = {i["id"]: i for i in json.load(open(os.path.join(GOLDEN, "page_figures.json")))["items"]}
    mib, gib = 2 ** 20, 2 ** 30
    for key, unit in (("score_bytes_8k", mib), ("prob_bytes_4k", mib), ("prob_bytes_128k", gib)):
        it = items[key]
        assert it["N"] ** 2 * it["elem_bytes"] == it["value"] * unit
    it = items["gemm_flops_per_exp_d128"]
    # one score element costs one exponential; the FLOP convention gives it 4d flops
    per_exp = oracle.flops_forward(1, 1, 1, it["d"], False)
    assert per_exp == it["value"]
    assert oracle.flops_backward(1, 1, 8, 64, True) == 2.5 * oracle.flops_forward(1, 1, 8, 64, True)


# ---------------------------------------------------------------- input recipe

def test_inputs_are_deterministic_and_bf16():
    a = inputs.draw_bf16(1, 2, 16, 8, 0)
    b = inputs.draw_bf16(1, 2, 16, 8, 0)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16
        assert torch.equal(x, y)
    c = inputs.draw_bf16(1, 2, 16, 8, 1)
    assert not torch.equal(a[0], c[0])


# ---------------------------------------------------------------- FP8 storage

@pytest.mark.parametrize("d", [64, 128])
def test_hadamard_is_orthogonal_with_plus_minus_entries(d):
    h = oracle.hadamard_matrix(d)
    np.testing.assert_allclose(h @ h.T, np.eye(d), rtol=0, atol=1e-13)
    assert np.all(np.abs(np.abs(h) * math.sqrt(d) - 1.0) < 1e-15)
    # Sylvester order: row 0 is constant, row 1 alternates sign
    assert np.all(h[0] > 0) and np.all(h[1, ::2] > 0) and np.all(h[1, 1::2] < 0)


def test_hadamard_rotation_leaves_attention_unchanged():
    q, k, v = rand_qkv(40, 64, 31)
    o1, l1, _ = oracle.head_forward(q, k, v, True, 0.125)
    o2, l2, _ = oracle.head_forward(oracle.rotate_rows(q), oracle.rotate_rows(k), v, True, 0.125)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


def test_hadamard_spreads_a_single_outlier():
    x = np.zeros((1, 128))
    x[0, 5] = 10.0
    y = oracle.rotate_rows(x)
    np.testing.assert_allclose(np.abs(y), 10.0 / math.sqrt(128), rtol=1e-15)


def test_e4m3_reference_quantiser():
    x = rng(32).standard_normal((64, 128)) * 3.0
    codes, delta = oracle.quantize_e4m3_reference(x)
    assert abs(delta - np.abs(x).max() / 448.0) < 1e-15
    deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * delta
    np.testing.assert_array_equal(oracle.dequantize_e4m3(codes, delta), deq)
    # the amax entry maps to 448 exactly; normals are within half an e4m3 ulp (2^-4 relative)
    assert abs(np.abs(deq).max() - np.abs(x).max()) <= 1e-12 * np.abs(x).max()
    big = np.abs(x) >= 2.0 ** -6 * delta
    assert np.all(np.abs(deq - x)[big] <= 2.0 ** -4 * np.abs(x)[big] + 1e-15)
    # e4m3 codes 0x7F / 0xFF are NaN: never produced
    assert not np.any((codes & 0x7F) == 0x7F)


def test_e4m3_blocks_one_block_is_the_per_tensor_quantiser():
    x = rng(33).standard_normal((2, 3, 50, 64)) * 2.0
    codes, deltas = oracle.quantize_e4m3_blocks_reference(x, 64)
    assert deltas.shape == (2, 3, 1)
    for b in range(2):
        for h in range(3):
            c1, d1 = oracle.quantize_e4m3_reference(x[b, h])
            np.testing.assert_array_equal(codes[b, h], c1)
            assert deltas[b, h, 0] == d1


def test_e4m3_blocks_are_independent_and_scale_covariant():
    x = rng(34).standard_normal((1, 1, 200, 128))
    codes, deltas = oracle.quantize_e4m3_blocks_reference(x, 64)
    assert deltas.shape == (1, 1, 4)  # 64 + 64 + 64 + 8 rows
    y = x.copy()
    y[..., 64:128, :] *= 2.0 ** 5  # one block scaled by a power of two
    codes2, deltas2 = oracle.quantize_e4m3_blocks_reference(y, 64)
    np.testing.assert_array_equal(codes2, codes)
    np.testing.assert_array_equal(deltas2[..., [0, 2, 3]], deltas[..., [0, 2, 3]])
    assert deltas2[0, 0, 1] == deltas[0, 0, 1] * 2.0 ** 5
    # the largest entry of each block is stored as +-448 exactly
    deq = oracle.dequantize_e4m3_blocks(codes, deltas, 64)
    for b, rows in enumerate([slice(0, 64), slice(64, 128), slice(128, 192), slice(192, 200)]):
        blk = x[..., rows, :]
        assert abs(np.abs(deq[..., rows, :]).max() - np.abs(blk).max()) <= 1e-12 * np.abs(blk).max()
        c = codes[..., rows, :]
        assert np.any((c & 0x7F) == 0x7E)  # 0x7E is 448


def test_e4m3_blocks_rounding_bound_and_zero_block():
    x = rng(35).standard_normal((1, 2, 256, 64)) * np.exp(rng(36).standard_normal((1, 2, 256, 1)) * 3)
    x[0, 1, 128:192] = 0.0
    codes, deltas = oracle.quantize_e4m3_blocks_reference(x, 64)
    assert deltas[0, 1, 2] == 1.0 and not np.any(codes[0, 1, 128:192])
    deq = oracle.dequantize_e4m3_blocks(codes, deltas, 64)
    dl = np.repeat(deltas, 64, axis=-1)[..., None]
    normal = np.abs(x) >= 2.0 ** -6 * dl
    # normals: half an ulp of a 3-bit mantissa; subnormals: half the spacing 2^-9 delta
    assert np.all(np.abs(deq - x)[normal] <= 2.0 ** -4 * np.abs(x)[normal] * (1 + 1e-12))
    assert np.all(np.abs(deq - x)[~normal] <= (2.0 ** -10 * dl * np.ones_like(x))[~normal] * (1 + 1e-12))
    # block scales follow the local magnitude
    amax = np.abs(x.reshape(1, 2, 4, 64, 64)).max(axis=(-2, -1))
    np.testing.assert_allclose(deltas, np.where(amax > 0, amax / 448.0, 1.0), rtol=1e-15)


# ---------------------------------------------------------------- sliding window

def test_window_covering_the_sequence_is_causal_attention():
    q, k, v, do = (t.double().numpy() for t in inputs.draw_fp32(1, 2, 30, 8, 13))
    o_c, l_c = oracle.forward(q, k, v, True, 0.3)
    for w in (30, 31, 100):
        o_w, l_w = oracle.forward_window(q, k, v, w, 0.3)
        np.testing.assert_array_equal(o_w, o_c)
        np.testing.assert_array_equal(l_w, l_c)
    dq, dk, dv = oracle.backward(q, k, v, do, True, 0.3)
    dq2, dk2, dv2 = oracle.backward_window(q, k, v, do, 30, 0.3)
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
        np.testing.assert_allclose(b, a, rtol=0, atol=1e-13)


def test_window_of_one_and_two_closed_forms():
    q, k, v, do = (t.double().numpy() for t in inputs.draw_fp32(1, 1, 12, 4, 14))
    s = 0.7
    # window 1: every query sees only its own key
    o, lse = oracle.forward_window(q, k, v, 1, s)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], s * np.einsum("nd,nd->n", q[0, 0], k[0, 0]), rtol=0, atol=1e-13)
    dq, dk, dv = oracle.backward_window(q, k, v, do, 1, s)
    np.testing.assert_allclose(dv, do, rtol=0, atol=1e-15)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    # window 2: a two-way softmax over keys i-1 and i
    o, _ = oracle.forward_window(q, k, v, 2, s)
    qq, kk, vv = q[0, 0], k[0, 0], v[0, 0]
    for i in range(1, 12):
        a, b = s * qq[i] @ kk[i - 1], s * qq[i] @ kk[i]
        w = 1.0 / (1.0 + math.exp(b - a))  # weight of key i-1
        np.testing.assert_allclose(o[0, 0, i], w * vv[i - 1] + (1 - w) * vv[i], rtol=0, atol=1e-13)


def test_window_backward_finite_differences():
    q, k, v, do = (t.double().numpy() for t in inputs.draw_fp32(1, 2, 10, 4, 15))
    k, v = k[:, :1], v[:, :1]  # two query heads share one key/value head
    w, s, h = 3, 0.5, 1e-6
    dq, dk, dv = oracle.backward_window(q, k, v, do, w, s)

    def loss(q_, k_, v_):
        return float((oracle.forward_window(q_, k_, v_, w, s)[0] * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 3, 1), (0, 0, 9, 2), (0, x.shape[1] - 1, 5, 0)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (loss(**{a + "_": b for a, b in args_p.items()}) - loss(**{a + "_": b for a, b in args_m.items()})) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


# ---------------------------------------------------------------- decode

def test_decode_is_the_last_row_of_causal_attention():
    # the token at position i attends keys 0..i: row i of causal attention
    q, k, v, _ = (t.double().numpy() for t in inputs.draw_fp32(1, 2, 40, 16, 9))
    o_c, l_c = oracle.forward(q, k, v, True, 0.25)
    for i in (0, 7, 39):
        o_d, l_d = oracle.decode(q[:, :, i], k[:, :, : i + 1], v[:, :, : i + 1], 0.25)
        np.testing.assert_allclose(o_d, o_c[:, :, i], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l_d, l_c[:, :, i], rtol=0, atol=1e-13)


def test_decode_closed_forms_and_groups():
    k = rng(40).standard_normal((2, 2, 33, 8))
    v = rng(41).standard_normal((2, 2, 33, 8))
    # q = 0: uniform weights, O = mean of V, L = ln N
    o, lse = oracle.decode(np.zeros((2, 4, 8)), k, v, 0.5)
    np.testing.assert_allclose(o, np.repeat(v.mean(axis=2), 2, axis=1), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(33.0), rtol=0, atol=1e-14)
    # query heads 2h and 2h+1 share key/value head h: same query, same row
    q = rng(42).standard_normal((2, 2, 8))
    o, lse = oracle.decode(np.repeat(q, 2, axis=1), k, v, 0.5)
    np.testing.assert_array_equal(o[:, 0], o[:, 1])
    np.testing.assert_array_equal(lse[:, 2], lse[:, 3])
    # one key dominating: O -> its value row
    kk = k.copy()
    kk[0, 0, 5] = 40.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    o, _ = oracle.decode(q, kk, v, 1.0)
    np.testing.assert_allclose(o[0, 0], v[0, 0, 5], rtol=0, atol=1e-8)


# ---------------------------------------------------------------- grouped-query attention

def test_gqa_with_one_query_head_per_kv_head_is_plain_attention():
    q, k, v, do = (t.double().numpy() for t in inputs.draw_fp32(1, 4, 24, 8, 5))
    o1, l1 = oracle.forward(q, k, v, True, 0.3)
    o2, l2 = oracle.forward_gqa(q, k, v, True, 0.3)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_gradients_by_central_differences(causal):
    # Two query heads share one key/value head: the gradient of the loss with
    # respect to the shared K and V must include both heads' contributions.
    r = rng(41)
    q = r.standard_normal((1, 2, 6, 4))
    k = r.standard_normal((1, 1, 6, 4))
    v = r.standard_normal((1, 1, 6, 4))
    do = r.standard_normal((1, 2, 6, 4))
    s, h = 0.5, 1e-6

    def loss(qq, kk, vv):
        o, _ = oracle.forward_gqa(qq, kk, vv, causal, s)
        return float((o * do).sum())

    dq, dk, dv = oracle.backward_gqa(q, k, v, do, causal, s)
    for x, g, idx in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        fd = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            xp = x.copy(); xp[pos] += h
            xm = x.copy(); xm[pos] -= h
            a_p = [q, k, v]; a_p[idx] = xp
            a_m = [q, k, v]; a_m[idx] = xm
            fd[pos] = (loss(*a_p) - loss(*a_m)) / (2 * h)
        assert np.abs(fd - g).max() <= 1e-6 * max(1.0, np.abs(g).max()), idx
