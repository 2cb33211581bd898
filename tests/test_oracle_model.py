"""Whole-forward pins of the oracle.

- Brute force on tiny shapes: an independent float64 NumPy statement with no
  cache and a materialised causal score matrix must agree with the oracle.
- The gates the Kipp pages fix: cached decode equals no-cache recomputation at
  every position ("Reproducing Kipp", section "Model-backed CPU and Metal
  gates"; "Kipp Model Support", section "What the gates check", Phase 2); the
  paged layout is bitwise equal to the contiguous one under permuted block
  tables and batched evaluation equals isolated evaluation ("Kipp Roadmap",
  status v0.0.2); truncate/resume replays ("Kipp Model Support", Phase 3).
- Invariants: the split of a prompt into rounds does not change the result,
  and logits never depend on later tokens (causality).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from synthetic import AFFINE4, BF16, Q8_0, Shape, make_block_permutation, make_tokens, make_weights

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")))

TINY = Shape("oracle-tiny", 2, 64, 4, 2, 16, 96, 128, True, rope_theta=1e4)
TINY_UNTIED = TINY.replace(name="oracle-tiny-untied", tied=False, n_layers=1)
TINY_Q8 = TINY.replace(name="oracle-tiny-q8", scheme=Q8_0, tied=False)
TINY_A4 = TINY.replace(name="oracle-tiny-affine4", scheme=AFFINE4, tied=False)
# Q8_0 blocks run along a head row, so the head width is a multiple of 32
TINY_KVQ8 = TINY.replace(name="oracle-tiny-kv-q8_0", head_dim=32, kv_quant=Q8_0)
KV_SHAPES = [TINY, TINY_KVQ8]            # the placement gates hold for either K/V storage


def _model(orc, shape, seed=7, threads=2):
    w = make_weights(shape, seed=seed)
    return orc.Model(shape, w, n_threads=threads), w


def _bf16r(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


def brute_force_logits(shape, w, tokens, weights64=None, kv_round=None):
    """float64 statement of the forward with no cache: every row's logits.
    kv_round maps K or V [T, n_kv, d] to its stored values (default: bf16)."""
    f = (lambda t: t.double().numpy()) if weights64 is None else weights64
    kv_round = _bf16r if kv_round is None else kv_round
    eps, d = shape.rms_eps, shape.head_dim
    T = len(tokens)
    x = w["embed"].double().numpy()[np.asarray(tokens)]

    def rms(v, g):
        return v / np.sqrt((v * v).mean(-1, keepdims=True) + eps) * g

    inv = shape.rope_theta ** (-np.arange(0, d, 2) / d)
    ang = np.arange(T)[:, None] * inv[None, :]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]

    def rope(v):
        a, b = v[..., : d // 2], v[..., d // 2:]
        return np.concatenate([a * cos - b * sin, b * cos + a * sin], -1)

    group = shape.n_q_heads // shape.n_kv_heads
    causal = np.triu(np.ones((T, T), bool), 1)
    for lw in w["layers"]:
        g = {k: lw[k].double().numpy() for k in ("attn_norm", "q_norm", "k_norm", "ffn_norm")}
        W = {k: f(lw[k]) for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")}
        h = rms(x, g["attn_norm"])
        q = (h @ W["wq"].T).reshape(T, shape.n_q_heads, d)
        k = (h @ W["wk"].T).reshape(T, shape.n_kv_heads, d)
        v = (h @ W["wv"].T).reshape(T, shape.n_kv_heads, d)
        q = rope(rms(q, g["q_norm"]))
        k = kv_round(rope(rms(k, g["k_norm"])))
        v = kv_round(v)
        k = np.repeat(k, group, axis=1)
        v = np.repeat(v, group, axis=1)
        s = np.einsum("thd,shd->hts", q, k) / math.sqrt(d)
        s[:, causal] = -np.inf
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        o = np.einsum("hts,shd->thd", p, v).reshape(T, -1)
        x = x + o @ W["wo"].T
        h = rms(x, g["ffn_norm"])
        a = h @ W["w_gate"].T
        x = x + (a / (1 + np.exp(-a)) * (h @ W["w_up"].T)) @ W["w_down"].T
    U = w["embed"] if shape.tied else w["lm_head"]
    return rms(x, w["final_norm"].double().numpy()) @ U.double().numpy().T


def _nmse(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(((a - b) ** 2).sum() / (b ** 2).sum())


@pytest.mark.parametrize("shape", [TINY, TINY_UNTIED], ids=lambda s: s.name)
def test_brute_force_agrees(orc, shape):
    m, w = _model(orc, shape)
    toks = make_tokens(11, shape.vocab, seed=5)
    got = m.session(max_ctx=64).eval(toks, all_rows=True)
    ref = brute_force_logits(shape, w, toks)
    for t in range(len(toks)):
        assert _nmse(got[t], ref[t]) < 1e-10, t
        assert int(np.argmax(got[t])) == int(np.argmax(ref[t]))


@pytest.mark.parametrize("shape", [TINY_Q8, TINY_A4], ids=lambda s: s.name)
def test_brute_force_agrees_quantized(orc, shape):
    """The quantized forward is the BF16 forward over the dequantised projections."""
    m, w = _model(orc, shape)
    toks = make_tokens(9, shape.vocab, seed=6)
    got = m.session(max_ctx=64).eval(toks, all_rows=True)
    unpack = orc.q8_0_unpack if shape.scheme == Q8_0 else orc.affine4_unpack
    deq = {}
    for l, lw in enumerate(w["layers"]):
        for name in orc.Model.PROJ:
            deq[id(lw[name])] = unpack(m.packed[l][name], lw[name].shape[1]).astype(np.float64)
    ref = brute_force_logits(shape, w, toks, weights64=lambda t: deq[id(t)])
    for t in range(len(toks)):
        assert _nmse(got[t], ref[t]) < 1e-10


def _q8_0_round(orc):
    """K or V [T, n_kv, d] as the Q8_0 cache stores it: FP32 rows packed in
    blocks of 32 by the oracle's (separately pinned) packer, then unpacked."""
    def rnd(a):
        a = np.asarray(a)
        f = np.ascontiguousarray(a.reshape(a.shape[0], -1), np.float32)
        return orc.q8_0_unpack(orc.q8_0_pack(f), f.shape[1]).astype(np.float64).reshape(a.shape)
    return rnd


def test_brute_force_agrees_q8_0_kv(orc):
    m, w = _model(orc, TINY_KVQ8)
    toks = make_tokens(11, TINY_KVQ8.vocab, seed=5)
    got = m.session(max_ctx=64).eval(toks, all_rows=True)
    ref = brute_force_logits(TINY_KVQ8, w, toks, kv_round=_q8_0_round(orc))
    for t in range(len(toks)):
        # a K/V value within FP32-vs-FP64 rounding of a quantization boundary may
        # take the neighbouring code on one side: 1e-8 leaves room for a few
        assert _nmse(got[t], ref[t]) < 1e-8, t
        assert int(np.argmax(got[t])) == int(np.argmax(ref[t]))


def test_q8_0_kv_cache_size_and_tolerance(orc):
    """About 1.9x smaller than bf16, and near the bf16-cache forward without equalling it."""
    kv = GOLD["q8_0_kv"]
    for key in ("4b", "14b"):
        s = __import__("synthetic").SHAPES[key]
        b16 = orc.kv_bytes_per_position(s)
        q8 = orc.kv_bytes_per_position(s.replace(kv_quant=Q8_0))
        assert b16 == 2 * s.n_kv_heads * s.head_dim * 2
        assert q8 == 2 * s.n_kv_heads * (s.head_dim // 32) * 34
        assert round(b16 / q8, 1) == kv["ratio_vs_bf16"]
    q, w = _model(orc, TINY_KVQ8)
    bf = orc.Model(TINY_KVQ8.replace(kv_quant=BF16), w, n_threads=2)
    toks = make_tokens(40, TINY.vocab, seed=12)
    got = q.session(max_ctx=64).eval(toks, all_rows=True)
    ref = bf.session(max_ctx=64).eval(toks, all_rows=True)
    e = _nmse(got, ref)
    assert 0 < e < kv["nmse_vs_bf16_cache"], e


def test_affine4_forward_stays_near_bf16(orc):
    """4-bit codes are lossy: the AFFINE4 forward is near the BF16 one, not equal."""
    a4, w = _model(orc, TINY_A4)
    bf = orc.Model(TINY_A4.replace(scheme=BF16), w, n_threads=2)
    toks = make_tokens(9, TINY_A4.vocab, seed=6)
    got = a4.session(max_ctx=64).eval(toks, all_rows=True)
    ref = bf.session(max_ctx=64).eval(toks, all_rows=True)
    e = _nmse(got, ref)
    assert 1e-6 < e < 1e-1, e


@pytest.mark.parametrize("shape", KV_SHAPES, ids=lambda s: s.name)
def test_cached_decode_equals_recompute(orc, shape):
    """Each position's K/V (bf16 or Q8_0) depends on that position only, so the
    cache a decode reads equals the one a full recompute builds."""
    tol = GOLD["nmse_cached_vs_recompute"]["value"]
    m, _ = _model(orc, shape)
    toks = make_tokens(40, shape.vocab, seed=8)
    full = m.session(max_ctx=64).eval(toks, all_rows=True)      # one round, no reuse
    s = m.session(max_ctx=64)
    s.eval(toks[:8])
    for t in range(8, 40):                                      # token by token from the cache
        got = s.eval(toks[t:t + 1])
        assert _nmse(got, full[t]) <= tol
        np.testing.assert_array_equal(got, full[t])             # the oracle is exact here
    assert s.pos == 40


@pytest.mark.parametrize("shape", KV_SHAPES, ids=lambda s: s.name)
def test_paged_equals_contiguous_under_permuted_tables(orc, shape):
    m, _ = _model(orc, shape)
    toks = make_tokens(100, shape.vocab, seed=9)
    ref = m.session(max_ctx=128).eval(toks, all_rows=True)
    for seed in (1, 2):
        pool = m.pool(16)
        s = m.session(pool=pool, max_ctx=128)
        s.set_block_table(make_block_permutation(16, seed)[:4])
        got = np.concatenate([s.eval(toks[:37], all_rows=True), s.eval(toks[37:38], all_rows=True),
                              s.eval(toks[38:], all_rows=True)])
        np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("shape", KV_SHAPES, ids=lambda s: s.name)
def test_batched_equals_isolated(orc, shape):
    m, _ = _model(orc, shape)
    pool = m.pool(32)
    prompts = [make_tokens(n, shape.vocab, seed=20 + n) for n in (5, 33, 12)]
    iso = []
    for p in prompts:
        s = m.session(max_ctx=128)
        iso.append([s.eval(p[:-1]), s.eval(p[-1:])])
    sess = [m.session(pool=pool, max_ctx=128) for _ in prompts]
    a = m.eval_batch(sess, [p[:-1] for p in prompts])
    b = m.eval_batch(sess, [p[-1:] for p in prompts])
    for i in range(3):
        np.testing.assert_array_equal(a[i], iso[i][0])
        np.testing.assert_array_equal(b[i], iso[i][1])


@pytest.mark.parametrize("shape", KV_SHAPES, ids=lambda s: s.name)
def test_chunking_and_causality(orc, shape):
    m, _ = _model(orc, shape)
    toks = make_tokens(50, shape.vocab, seed=10)
    one = m.session(max_ctx=64).eval(toks, all_rows=True)
    s = m.session(max_ctx=64)
    parts = [s.eval(toks[a:b], all_rows=True) for a, b in ((0, 5), (5, 45), (45, 50))]
    np.testing.assert_array_equal(np.concatenate(parts), one)
    toks2 = toks.copy()
    toks2[30:] = (toks2[30:] + 1) % shape.vocab                  # change only later tokens
    two = m.session(max_ctx=64).eval(toks2, all_rows=True)
    np.testing.assert_array_equal(two[:30], one[:30])
    assert not np.array_equal(two[30], one[30])


@pytest.mark.parametrize("shape", KV_SHAPES, ids=lambda s: s.name)
def test_truncate_and_resume(orc, shape):
    m, _ = _model(orc, shape)
    toks = make_tokens(30, shape.vocab, seed=11)
    s = m.session(max_ctx=64)
    ref = s.eval(toks, all_rows=True)
    s.truncate(12)
    assert s.pos == 12
    np.testing.assert_array_equal(s.eval(toks[12:20], all_rows=True), ref[12:20])


def test_capacity_errors(orc):
    m, _ = _model(orc, TINY)
    s = m.session(max_ctx=16)
    with pytest.raises(RuntimeError):
        s.eval(make_tokens(17, TINY.vocab, seed=1))
    # a Q8_0 cache needs whole 32-value blocks per head row
    with pytest.raises(ValueError):
        orc.Model(TINY.replace(kv_quant=Q8_0), make_weights(TINY, seed=7), n_threads=1)
    with pytest.raises(RuntimeError):
        s.eval(np.array([TINY.vocab], np.int32))
    pool = m.pool(1)
    s = m.session(pool=pool, max_ctx=128)
    s.eval(make_tokens(32, TINY.vocab, seed=2))
    with pytest.raises(RuntimeError):
        s.eval(make_tokens(1, TINY.vocab, seed=3))


def test_shapes_follow_the_registry(orc):
    import synthetic
    for key in ("0.6b", "4b", "8b-q8_0", "14b"):
        s = synthetic.SHAPES[key]
        assert s.vocab == GOLD["vocab"]["value"]
        assert s.n_kv_heads == GOLD["n_kv_heads"]["value"]
        assert s.head_dim == GOLD["head_dim"]["value"]
        assert s.rms_eps == GOLD["rms_eps"]["value"]
    s = synthetic.SHAPES["0.6b"]
    assert (s.q_width, s.hidden) == (GOLD["attn_width_0p6b"]["value"], GOLD["attn_width_0p6b"]["hidden"])
    assert 34 * 8 / 32 == GOLD["q8_0"]["bits_per_weight"] and orc.Q8_0_BYTES == 34
    a4 = GOLD["affine4_gs32"]
    assert orc.AFFINE4_BYTES * 8 / a4["weights_per_group"] == a4["bits_per_weight"]
    assert orc.AFFINE4_BYTES == (a4["weights_per_group"] * a4["code_bits"] + 2 * 16) // 8
    assert orc.BLOCK == GOLD["kv_block_positions"]["value"]
    assert BF16 == 0


@pytest.mark.parametrize("shape", KV_SHAPES, ids=lambda s: s.name)
def test_selected_rows_and_append_only(orc, shape):
    """eval_rows returns exactly the listed rows of the every-row logits, and a
    round appended without logits leaves the same cache as one that computed
    them (the full-size GPU gates lean on both: they score a sample of the
    rows of a long round, and prefill long prior contexts with append)."""
    m, _ = _model(orc, shape)
    toks = make_tokens(70, shape.vocab, seed=12)
    full = m.session(max_ctx=128).eval(toks, all_rows=True)
    rows = [0, 5, 31, 32, 63, 69]
    got = m.session(max_ctx=128).eval_rows(toks, rows)
    np.testing.assert_array_equal(got, full[rows])
    s = m.session(max_ctx=128)
    s.append(toks[:64])
    assert s.pos == 64
    np.testing.assert_array_equal(s.eval(toks[64:], all_rows=True), full[64:])
    with pytest.raises(RuntimeError):
        m.session(max_ctx=128).eval_rows(toks[:10], [3, 3])        # rows must increase
    with pytest.raises(RuntimeError):
        m.session(max_ctx=128).eval_rows(toks[:10], [10])          # and lie in the round
