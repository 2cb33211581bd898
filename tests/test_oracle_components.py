"""Pins of the oracle's layer components against closed forms and invariants.

Each test is chosen so that a plausible slip in the oracle (eps outside the
root, a gain read as 1 + g, a RoPE sign or pairing error, a wrong softmax
scale, the wrong GQA grouping, a transposed weight) makes it fail.
"""
import math

import numpy as np
import torch

EPS = 1e-6


def _bits(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def test_rmsnorm_closed_form(orc):
    # x = c * ones: mean(x^2) = c^2, so y = c / sqrt(c^2 + eps) * g exactly
    for c in (0.5, 1e-3, 3.0, -2.0):
        g = np.array([1.0, 2.0, 0.5, -1.0] * 16, np.float32)      # exact in bf16
        y = orc.rmsnorm(np.full(64, c, np.float32), _bits(g), EPS)
        want = c / math.sqrt(c * c + EPS) * g.astype(np.float64)
        np.testing.assert_allclose(y, want, rtol=1e-7, atol=0)
    # eps inside the root: tiny inputs are damped, not amplified
    y = orc.rmsnorm(np.full(8, 1e-4, np.float32), _bits(np.ones(8)), EPS)
    np.testing.assert_allclose(y, 1e-4 / math.sqrt(1e-8 + 1e-6), rtol=1e-6)


def test_rmsnorm_unit_gain_gives_unit_rms(orc):
    rng = np.random.default_rng(0)
    x = rng.standard_normal(1024).astype(np.float32) * 7
    y = orc.rmsnorm(x, _bits(np.ones(1024)), EPS)
    rms = math.sqrt(float((y.astype(np.float64) ** 2).mean()))
    assert abs(rms - 1.0) < 1e-6
    # scale invariance (up to eps) and linearity in the gain
    y2 = orc.rmsnorm(x * 4, _bits(np.full(1024, 2.0)), EPS)
    np.testing.assert_allclose(y2, 2 * y, rtol=1e-5)


def test_rope_closed_form_basis_vectors(orc):
    d, theta = 16, 10000.0
    for pos in (0, 1, 5, 1000):
        for i in range(d // 2):
            e = np.zeros(d, np.float32)
            e[i] = 1.0
            a = pos * theta ** (-2.0 * i / d)
            out = orc.rope(e, pos, theta)
            want = np.zeros(d)
            want[i], want[i + d // 2] = math.cos(a), math.sin(a)     # e_i -> cos e_i + sin e_{i+d/2}
            np.testing.assert_allclose(out, want, atol=1e-7)
            e2 = np.zeros(d, np.float32)
            e2[i + d // 2] = 1.0
            want2 = np.zeros(d)
            want2[i], want2[i + d // 2] = -math.sin(a), math.cos(a)
            np.testing.assert_allclose(orc.rope(e2, pos, theta), want2, atol=1e-7)


def test_rope_identity_norm_and_relative_position(orc):
    rng = np.random.default_rng(1)
    d, theta = 128, 1e6
    q = rng.standard_normal(d).astype(np.float32)
    k = rng.standard_normal(d).astype(np.float32)
    np.testing.assert_array_equal(orc.rope(q, 0, theta), q)
    r = orc.rope(q, 777, theta)
    assert abs(np.linalg.norm(r.astype(np.float64)) - np.linalg.norm(q.astype(np.float64))) < 1e-5
    # <rope(q, m), rope(k, n)> depends only on m - n
    for m, n in ((10, 3), (1010, 1003), (16000, 15993)):
        dot = float(orc.rope(q, m, theta).astype(np.float64) @ orc.rope(k, n, theta))
        ref = float(orc.rope(q, 7, theta).astype(np.float64) @ orc.rope(k, 0, theta))
        assert abs(dot - ref) < 2e-4 * d ** 0.5


def test_silu_closed_form(orc):
    assert orc.silu(0.0) == 0.0
    for z in (0.3, 1.0, 2.5, 7.0):
        assert abs(orc.silu(z) - orc.silu(-z) - z) < 1e-6 * max(1, z)
        assert abs(orc.silu(z) - z / (1 + math.exp(-z))) < 1e-7 * max(1, z)
    assert orc.silu(40.0) == np.float32(40.0)


def test_matmul_orientation_and_values(orc):
    rng = np.random.default_rng(2)
    n_out, n_in = 48, 96
    W = torch.randn(n_out, n_in, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    Wb = W.view(torch.int16).numpy().view(np.uint16)
    Wf = W.float().numpy().astype(np.float64)
    # unit inputs pick out columns: y[o] = W[o][i]
    for i in (0, 17, 95):
        e = np.zeros(n_in, np.float32)
        e[i] = 1.0
        np.testing.assert_array_equal(orc.matmul(Wb, 0, n_out, n_in, e)[0], Wf[:, i].astype(np.float32))
    x = rng.standard_normal((5, n_in)).astype(np.float32)
    y = orc.matmul(Wb, 0, n_out, n_in, x, n_threads=3)
    np.testing.assert_allclose(y, x.astype(np.float64) @ Wf.T, rtol=1e-6, atol=1e-6)
    # Q8_0 weights: the product with the dequantised matrix
    packed = orc.q8_0_pack(Wf.astype(np.float32))
    deq = orc.q8_0_unpack(packed, n_in).astype(np.float64)
    yq = orc.matmul(packed, 1, n_out, n_in, x, n_threads=2)
    np.testing.assert_allclose(yq, x.astype(np.float64) @ deq.T, rtol=1e-6, atol=1e-6)
    # AFFINE4_GS32 weights: the same, with 20-byte groups along each row
    groups = orc.affine4_pack(Wf.astype(np.float32))
    assert groups.shape == (n_out, n_in // 32 * 20)
    deq4 = orc.affine4_unpack(groups, n_in).astype(np.float64)
    for i in (0, 17, 95):
        e = np.zeros(n_in, np.float32)
        e[i] = 1.0
        np.testing.assert_array_equal(orc.matmul(groups, 2, n_out, n_in, e)[0],
                                      deq4[:, i].astype(np.float32))
    y4 = orc.matmul(groups, 2, n_out, n_in, x, n_threads=2)
    np.testing.assert_allclose(y4, x.astype(np.float64) @ deq4.T, rtol=1e-6, atol=1e-6)


def _kv(a):
    return _bits(a).reshape(np.asarray(a).shape)


def test_attention_single_key_and_constant_values(orc):
    rng = np.random.default_rng(4)
    n_q, n_kv, d = 4, 2, 8
    q = rng.standard_normal((n_q, d)).astype(np.float32)
    K = _kv(rng.standard_normal((1, n_kv, d)))
    V = _kv(rng.standard_normal((1, n_kv, d)))
    o = orc.gqa_attend(q, K, V, n_q, n_kv, d)
    Vf = torch.from_numpy(V.view(np.int16)).view(torch.bfloat16).float().numpy()
    for h in range(n_q):                         # one key: o = V exactly
        np.testing.assert_array_equal(o[h], Vf[0, h // 2])
    # identical V rows give that row, whatever the keys
    ctx = 9
    K = _kv(rng.standard_normal((ctx, n_kv, d)))
    row = rng.standard_normal((1, n_kv, d))
    V = _kv(np.repeat(row, ctx, axis=0))
    o = orc.gqa_attend(q, K, V, n_q, n_kv, d)
    Vf = torch.from_numpy(V.view(np.int16)).view(torch.bfloat16).float().numpy()
    for h in range(n_q):
        np.testing.assert_array_equal(o[h], Vf[0, h // 2])


def test_attention_uniform_scores_give_mean_and_two_key_weights(orc):
    rng = np.random.default_rng(5)
    n_q, n_kv, d, ctx = 2, 1, 16, 6
    q = rng.standard_normal((n_q, d)).astype(np.float32)
    Vr = rng.standard_normal((ctx, n_kv, d))
    V = _kv(Vr)
    Vf = torch.from_numpy(V.view(np.int16)).view(torch.bfloat16).double().numpy()
    o = orc.gqa_attend(q, _kv(np.zeros((ctx, n_kv, d))), V, n_q, n_kv, d)
    np.testing.assert_allclose(o[0], Vf[:, 0].mean(0), rtol=1e-6, atol=1e-7)
    # two keys along e_0 with scores a/sqrt(d), b/sqrt(d): weights by hand
    q = np.zeros((1, d), np.float32)
    q[0, 0] = 1.0
    K = np.zeros((2, 1, d))
    K[0, 0, 0], K[1, 0, 0] = 2.0, -1.0
    V = np.zeros((2, 1, d))
    V[0, 0, 1], V[1, 0, 1] = 1.0, 0.0
    o = orc.gqa_attend(q, _kv(K), _kv(V), 1, 1, d)
    s0, s1 = 2.0 / math.sqrt(d), -1.0 / math.sqrt(d)
    w0 = math.exp(s0) / (math.exp(s0) + math.exp(s1))
    assert abs(o[0, 1] - w0) < 1e-7 and o[0, 0] == 0.0


def test_attention_gqa_grouping_is_contiguous(orc):
    # V of KV head j is the constant j + 1: query head h must read KV head h // (n_q / n_kv)
    n_q, n_kv, d, ctx = 8, 2, 4, 5
    rng = np.random.default_rng(6)
    V = np.zeros((ctx, n_kv, d))
    for j in range(n_kv):
        V[:, j, :] = j + 1
    o = orc.gqa_attend(rng.standard_normal((n_q, d)).astype(np.float32),
                       _kv(rng.standard_normal((ctx, n_kv, d))), _kv(V), n_q, n_kv, d)
    for h in range(n_q):
        np.testing.assert_allclose(o[h], h // 4 + 1, rtol=1e-7)
