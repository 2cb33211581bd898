"""The opt-in Q8_0 K/V cache on the CUDA path ("Kipp Roadmap", status v0.0.4
and "Delivered since": an opt-in Q8_0 KV cache, about 1.9x smaller than BF16,
gated for tolerance and placement invariance).

- The cache writers' packing equals the oracle's Q8_0 packer bit for bit
  (operator gate q3_op_kv_pack_q8_0 on random and edge rows: all-zero
  blocks, exact multiples of the scale with ties, signed zeros, wide ranges).
- A position's K/V take 2 * n_kv * 136 bytes a layer, as the oracle counts
  them: 1.88x smaller than BF16.
- The forward against the oracle's Q8_0-cache forward (the usual gate:
  NMSE <= 1e-4, identical argmax): prompt and greedy decode over a permuted
  table, chunked prompts crossing block edges, batched decode over long
  unequal contexts (split-KV merges), and the Qwen3-4B heads at a 2,000
  position context.
- Placement invariance: a permuted block table gives the identity table's
  logits bit for bit.
"""
import numpy as np
import pytest
import torch

import synthetic
from helpers import Pair, check_row, make_shape

pytestmark = pytest.mark.gpu

TINY_Q8KV = make_shape("tiny", kv_quant=synthetic.Q8_0, name="tiny-kv-q8_0")


@pytest.fixture(scope="module")
def q3():
    import qwen3_dense_decoder_gb300 as q3
    q3.build()
    return q3


@pytest.fixture(scope="module")
def pair():
    return Pair(TINY_Q8KV, seed=801, max_ctx=512, max_round_tokens=256, n_blocks=96)


def _rows_with_edges(n, seed):
    g = torch.Generator().manual_seed(seed)
    r = torch.randn(n, 128, generator=g) * torch.logspace(-3, 2, n).unsqueeze(1)
    r[0, :32] = 0.0                                         # an all-zero block
    r[0, 32:64] = -0.0                                      # signed zeros
    r[1, :32] = torch.arange(-16, 16, dtype=torch.float32) * (3.0 / 127)   # multiples of d
    r[2, :32] = torch.tensor([(k + 0.5) * 0.25 for k in range(-16, 16)])   # halfway codes
    r[2, 0] = 127 * 0.25                                    # pins d = 0.25 for those ties
    r[3, :] = 1e-30                                         # a range below the fp16 scale's
    r[4, 64:96] = 6.5e4                                     # near the fp16 top
    return r.contiguous()


def test_kv_packing_matches_oracle_packer_bitwise(q3, orc):
    rows = _rows_with_edges(300, 3)
    got = q3.op_kv_pack_q8_0(rows.cuda()).cpu().numpy()
    ref = orc.q8_0_pack(rows.numpy())
    assert got.shape == ref.shape == (300, 136)
    np.testing.assert_array_equal(got, ref)


def test_bytes_per_position_follow_the_oracle(q3, orc, pair):
    assert pair.model.kv_bytes_per_position == orc.kv_bytes_per_position(TINY_Q8KV) == 2 * 8 * 136
    bf16 = 2 * 8 * 128 * 2
    assert round(bf16 / pair.model.kv_bytes_per_position, 1) == 1.9      # the pages' "about 1.9x"


def _run(pair, g, o, rounds, n_decode, tag):
    for r in rounds:
        got, ref, am = pair.eval(g, o, r)
        c = check_row(got, ref, f"{tag}/prefill{len(r)}")
        assert c.ok, (tag, len(r), c)
    tok = c.argmax_ref
    for step in range(n_decode):
        got, ref, am = pair.eval(g, o, [tok])
        c = check_row(got, ref, f"{tag}/decode")
        assert c.ok, (tag, step, c)
        assert am == c.argmax_gpu
        tok = c.argmax_ref


def test_prompt_then_greedy_decode_permuted_table(pair):
    assert not pair.model.fused_decode and not pair.model.prefill_tc   # per-op decode, mma.sync prefill
    perm = synthetic.make_block_permutation(96, seed=802)
    g, o = pair.sessions(table=perm[:4])
    _run(pair, g, o, [synthetic.make_tokens(8, TINY_Q8KV.vocab, seed=803)], 8, "kvq8/tiny")
    g.close()


def test_chunked_prompt_across_block_edges(pair):
    perm = synthetic.make_block_permutation(96, seed=804)
    g, o = pair.sessions(table=perm[20:32])
    toks = synthetic.make_tokens(280, TINY_Q8KV.vocab, seed=805)
    _run(pair, g, o, [toks[:256], toks[256:]], 20, "kvq8/tiny-300")
    g.close()


def test_paged_equals_identity_table_bitwise(pair):
    prompt = synthetic.make_tokens(70, TINY_Q8KV.vocab, seed=806)
    outs = []
    for table in (np.arange(40, 43), synthetic.make_block_permutation(96, seed=807)[50:53]):
        g = pair.pool.session()
        g.set_block_table(table)
        rows = []
        for toks in (prompt[:45], prompt[45:], [5], [6], [7]):
            g.eval(torch.tensor(np.asarray(toks, np.int32), device="cuda"), pair.logits[0])
            pair.model.sync()
            rows.append(pair.logits[0].cpu().numpy().copy())
        outs.append(np.stack(rows))
        g.close()
    np.testing.assert_array_equal(outs[0], outs[1])


def test_batched_decode_over_long_unequal_contexts():
    pair = Pair(TINY_Q8KV, seed=808, max_ctx=3200, max_round_tokens=256, n_blocks=220, max_sessions=4)
    lens = [300, 1700, 3100]
    perm = synthetic.make_block_permutation(220, seed=809)
    tables = [perm[0:60], perm[60:120], None]
    gs, os_, nxt = [], [], []
    for i, n in enumerate(lens):
        g, o = pair.sessions(table=tables[i])
        toks = synthetic.make_tokens(n, TINY_Q8KV.vocab, seed=810 + i)
        for a in range(0, n, 256):
            got, ref, _ = pair.eval(g, o, toks[a:a + 256])
        assert check_row(got, ref, f"kvq8/long/{n}").ok, i
        gs.append(g)
        os_.append(o)
        nxt.append(int(np.argmax(ref)))
    for step in range(4):
        got, ref, am = pair.eval_batch(gs, os_, [[t] for t in nxt])
        for i in range(3):
            c = check_row(got[i], ref[i], f"kvq8/long-batched/{lens[i]}")
            assert c.ok, (step, i, c)
            assert am[i] == c.argmax_gpu
        nxt = [int(np.argmax(r)) for r in ref]
    for g in gs:
        g.close()


def test_qwen3_4b_heads_batched_decode_at_2000_positions():
    shape = make_shape("4b", n_layers=1, kv_quant=synthetic.Q8_0, name="qwen3-4b-kv-q8_0")
    B, n = 6, 2000
    pair = Pair(shape, seed=820, max_ctx=n + 64, max_round_tokens=2048, n_blocks=B * 66 + 8,
                max_sessions=B + 2)
    gs, os_ = [], []
    for i in range(B):
        g, o = pair.sessions()
        toks = synthetic.make_tokens(n - 37 * i, shape.vocab, seed=821 + i)
        g.eval(torch.tensor(toks, device="cuda"), pair.logits[0])
        o.append(toks)
        gs.append(g)
        os_.append(o)
    pair.model.sync()
    nxt = [[int(t)] for t in synthetic.make_tokens(B, shape.vocab, seed=830)]
    for step in range(3):
        got, ref, am = pair.eval_batch(gs, os_, nxt)
        for i in range(B):
            c = check_row(got[i], ref[i], "kvq8/4b-b6")
            assert c.ok, (step, i, c)
        nxt = [[int(np.argmax(r))] for r in ref]
    for g in gs:
        g.close()
