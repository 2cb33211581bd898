"""Whole-forward parity of the CUDA path against the oracle (the pages' Phase 3
and Phase 4 gates: "Kipp Model Support", sections "What the gates check" and
"CUDA (NVIDIA H100 80GB ...)"): identical argmax and full-logit NMSE <= 1e-4
at prefill and at every decode position, truncate/resume, reset/reuse and
batched-equals-isolated evaluation; paged KV bitwise equal to an identity
block table ("Kipp Roadmap", status v0.0.2).  Decode is teacher-forced: both
sides consume the oracle's greedy token.
"""
import numpy as np
import pytest
import torch

import synthetic
from helpers import NMSE_BOUND, Pair, check_row, make_shape

pytestmark = pytest.mark.gpu

TINY = make_shape("tiny")


@pytest.fixture(scope="module")
def tiny_pair():
    return Pair(TINY, seed=101, max_ctx=512, max_round_tokens=256, n_blocks=96)


def _run(pair, g, o, rounds, n_decode, tag=""):
    """Prefill rounds then greedy decode; every row checked.  Returns the checks."""
    checks = []
    for r in rounds:
        got, ref, am = pair.eval(g, o, r)
        c = check_row(got, ref, f"{tag}/prefill{len(r)}")
        assert am == c.argmax_gpu
        checks.append(c)
        assert c.ok, (tag, "prefill", len(r), c)
    tok = checks[-1].argmax_ref
    for step in range(n_decode):
        got, ref, am = pair.eval(g, o, [tok])
        c = check_row(got, ref, f"{tag}/decode")
        assert am == c.argmax_gpu
        checks.append(c)
        assert c.ok, (tag, "decode", step, c)
        tok = c.argmax_ref
    return checks


def test_tiny_prompt_then_greedy_decode_permuted_table(tiny_pair):
    perm = synthetic.make_block_permutation(96, seed=7)
    g, o = tiny_pair.sessions(table=perm[:4])
    prompt = synthetic.make_tokens(8, TINY.vocab, seed=11)
    checks = _run(tiny_pair, g, o, [prompt], 8, "tiny")
    assert max(c.nmse for c in checks) <= NMSE_BOUND
    assert g.pos == o.pos == 16


def test_tiny_multi_block_context(tiny_pair):
    # 280-token prompt: chunked into 256 + 24 rows; decode crosses the block edge at 288
    perm = synthetic.make_block_permutation(96, seed=8)
    g, o = tiny_pair.sessions(table=perm[10:20])
    prompt = synthetic.make_tokens(280, TINY.vocab, seed=12)
    _run(tiny_pair, g, o, [prompt], 20, "tiny-300")
    assert g.pos == 300


def test_paged_equals_identity_table_bitwise(tiny_pair):
    prompt = synthetic.make_tokens(70, TINY.vocab, seed=13)
    outs = []
    for table in (np.arange(40, 43), synthetic.make_block_permutation(96, seed=9)[50:53]):
        g = tiny_pair.pool.session()
        g.set_block_table(table)
        rows = []
        for toks in (prompt[:45], prompt[45:], [5], [6], [7]):
            t = torch.tensor(np.asarray(toks, np.int32), device="cuda")
            g.eval(t, tiny_pair.logits[0])
            tiny_pair.model.sync()
            rows.append(tiny_pair.logits[0].cpu().numpy().copy())
        outs.append(np.stack(rows))
        g.close()
    np.testing.assert_array_equal(outs[0], outs[1])


def test_batched_equals_isolated(tiny_pair):
    prompts = [synthetic.make_tokens(n, TINY.vocab, seed=30 + n) for n in (5, 33, 12)]
    # isolated, on the GPU
    iso = []
    for p in prompts:
        g = tiny_pair.pool.session()
        t = torch.tensor(p, device="cuda")
        g.eval(t, tiny_pair.logits[0])
        tiny_pair.model.sync()
        iso.append(tiny_pair.logits[0].cpu().numpy().copy())
        g.close()
    # batched, against the oracle and against isolated
    gs, os_ = zip(*[tiny_pair.sessions() for _ in prompts])
    got, ref, am = tiny_pair.eval_batch(list(gs), list(os_), prompts)
    for i in range(3):
        c = check_row(got[i], ref[i])
        assert c.ok, (i, c)
        assert am[i] == c.argmax_gpu
        assert check_row(got[i], iso[i]).nmse <= NMSE_BOUND
    # a batched decode round: one token per session
    toks = [[int(np.argmax(ref[i]))] for i in range(3)]
    got, ref, am = tiny_pair.eval_batch(list(gs), list(os_), toks)
    for i in range(3):
        assert check_row(got[i], ref[i]).ok
    for g in gs:
        g.close()


def test_prefill_head_epilogue_and_split_fallback(tiny_pair):
    """Prefill rounds of the BF16 cache apply the q/k head norm, RoPE and the
    K/V append in the QKV GEMM's epilogue when its plan does not split K (70
    tokens: 32-token tiles with a 6-token tail; 170: 64-token tiles with a
    42-token tail) and in the separate kernel when it does (20 tokens, four K
    splits).  Each matches the oracle, and batched decode rounds read back the
    K/V each one wrote."""
    m = tiny_pair.model
    separate = {}
    gs, os_ = [], []
    for n in (20, 70, 170):
        g, o = tiny_pair.sessions()
        toks = synthetic.make_tokens(n, TINY.vocab, seed=900 + n)
        m.profile(True)
        m.profile_reset()
        got, ref, am = tiny_pair.eval(g, o, toks)
        separate[n] = m.profile_read()["qk_norm_rope_append"][1]
        m.profile(False)
        c = check_row(got, ref, f"tiny/head-epilogue/prefill{n}")
        assert c.ok, (n, c)
        assert am == c.argmax_gpu
        gs.append(g)
        os_.append(o)
    assert separate == {20: TINY.n_layers, 70: 0, 170: 0}, separate
    nxt = [[int(t)] for t in synthetic.make_tokens(3, TINY.vocab, seed=950)]
    for step in range(3):
        got, ref, am = tiny_pair.eval_batch(gs, os_, nxt)
        for i in range(3):
            c = check_row(got[i], ref[i], "tiny/head-epilogue/decode")
            assert c.ok, (step, i, c)
            assert am[i] == c.argmax_gpu
        nxt = [[int(np.argmax(r))] for r in ref]
    for g in gs:
        g.close()


def test_batched_decode_over_long_unequal_contexts():
    # three sessions of 300, 1,700 and 3,100 positions decode together: the
    # attention's split count follows the longest row, shorter rows leave
    # splits empty, and each row's splits merge in order
    pair = Pair(TINY, seed=131, max_ctx=3200, max_round_tokens=256, n_blocks=220, max_sessions=4)
    lens = [300, 1700, 3100]
    perm = synthetic.make_block_permutation(220, seed=140)
    tables = [perm[0:60], perm[60:120], None]                 # disjoint; the third from the allocator
    gs, os_, nxt = [], [], []
    for i, n in enumerate(lens):
        g, o = pair.sessions(table=tables[i])
        toks = synthetic.make_tokens(n, TINY.vocab, seed=150 + i)
        for a in range(0, n, 256):
            got, ref, _ = pair.eval(g, o, toks[a:a + 256])
        assert check_row(got, ref).ok, i
        gs.append(g)
        os_.append(o)
        nxt.append(int(np.argmax(ref)))
    for step in range(4):
        got, ref, am = pair.eval_batch(gs, os_, [[t] for t in nxt])
        for i in range(3):
            c = check_row(got[i], ref[i], f"long-batched/{lens[i]}")
            assert c.ok, (step, i, c)
            assert am[i] == c.argmax_gpu
        nxt = [int(np.argmax(r)) for r in ref]
    for g in gs:
        g.close()


def test_truncate_resume_and_reset_reuse(tiny_pair):
    prompt = synthetic.make_tokens(40, TINY.vocab, seed=14)
    g, o = tiny_pair.sessions()
    first, _, _ = tiny_pair.eval(g, o, prompt[:30])
    g.truncate(12)
    o.truncate(12)
    assert g.pos == 12
    got, ref, _ = tiny_pair.eval(g, o, prompt[12:20])
    assert check_row(got, ref).ok
    g.reset()
    assert g.pos == 0
    t = torch.tensor(prompt[:30], device="cuda")
    g.eval(t, tiny_pair.logits[0])
    tiny_pair.model.sync()
    np.testing.assert_array_equal(tiny_pair.logits[0].cpu().numpy(), first)   # stateless prefill
    g.close()


def test_bad_token_is_a_device_check_and_poisons(orc):
    import qwen3_dense_decoder_gb300 as q3
    pair = Pair(TINY.replace(n_layers=1), seed=5, max_ctx=64, max_round_tokens=32, n_blocks=4)
    g = pair.pool.session()
    bad = torch.tensor([1, TINY.vocab + 3], dtype=torch.int32, device="cuda")
    g.eval(bad, pair.logits[0])
    with pytest.raises(q3.Q3Error) as e:
        pair.model.sync()
    assert e.value.code == -7
    with pytest.raises(q3.Q3Error) as e:
        g.eval(bad[:1], pair.logits[0])
    assert e.value.code == -8


def test_capacity_errors_are_host_side(orc):
    import qwen3_dense_decoder_gb300 as q3
    pair = Pair(TINY.replace(n_layers=1), seed=6, max_ctx=64, max_round_tokens=32, n_blocks=2)
    g = pair.pool.session()
    t = torch.zeros(65, dtype=torch.int32, device="cuda")
    with pytest.raises(q3.Q3Error) as e:
        g.eval(t, pair.logits[0])
    assert e.value.code == -5                       # CTX_OVERFLOW
    g.eval(t[:64], pair.logits[0])                  # fills both blocks
    pair.model.sync()
    g2 = pair.pool.session()
    with pytest.raises(q3.Q3Error) as e:
        g2.eval(t[:1], pair.logits[0])
    assert e.value.code == -4                       # POOL_EXHAUSTED


def test_qwen3_0p6b_ragged_three_round_prefill():
    shape = make_shape("0.6b")
    pair = Pair(shape, seed=202, max_ctx=256, max_round_tokens=128, n_blocks=16)
    perm = synthetic.make_block_permutation(16, seed=3)
    g, o = pair.sessions(table=perm[:5])
    prompt = synthetic.make_tokens(128, shape.vocab, seed=21)
    _run(pair, g, o, [prompt[:5], prompt[5:45], prompt[45:128]], 4, "0.6b")


def test_qwen3_8b_q8_0_shape_two_layers():
    shape = make_shape("8b-q8_0", n_layers=2)
    pair = Pair(shape, seed=303, max_ctx=128, max_round_tokens=64, n_blocks=8)
    g, o = pair.sessions(table=synthetic.make_block_permutation(8, seed=4)[:2])
    prompt = synthetic.make_tokens(16, shape.vocab, seed=22)
    _run(pair, g, o, [prompt], 4, "8b-q8_0")


def test_qwen3_4b_affine4_shape_two_layers():
    """AFFINE4_GS32 projections: both sides quantize the same bf16 weights
    (bit-equal packers), so the gate is the usual one against the oracle's
    AFFINE4 forward; one-token decode rounds take the tensor-core path."""
    shape = make_shape("4b", n_layers=2, scheme=synthetic.AFFINE4, name="qwen3-4b-affine4")
    pair = Pair(shape, seed=505, max_ctx=128, max_round_tokens=64, n_blocks=8)
    g, o = pair.sessions(table=synthetic.make_block_permutation(8, seed=6)[:3])
    prompt = synthetic.make_tokens(40, shape.vocab, seed=24)
    _run(pair, g, o, [prompt[:7], prompt[7:40]], 4, "4b-affine4")
    assert not pair.model.fused_decode


def test_qwen3_4b_shape_full_depth():
    shape = make_shape("4b")
    pair = Pair(shape, seed=404, max_ctx=128, max_round_tokens=64, n_blocks=8)
    g, o = pair.sessions(table=synthetic.make_block_permutation(8, seed=5)[:2])
    prompt = synthetic.make_tokens(24, shape.vocab, seed=23)
    _run(pair, g, o, [prompt], 3, "4b")
