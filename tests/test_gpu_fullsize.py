"""Parity at the sizes the benchmark runs: the same kernels, tile plans,
split-K choices and attention schedules as the timed paths, against the
oracle (the pages' model-backed gates: "Reproducing Kipp", section
"Model-backed CPU and Metal gates"; "Kipp Model Support", section "What the
gates check": identical argmax and full-logit NMSE <= 1e-4 per row).

- One 2,048-token round of the Qwen3-4B shape (2 layers) in a model built
  with max_round_tokens = 2048, as the prefill benchmark builds it; every
  64th row and the last scored through q3_session_eval_n, and the last row
  again through q3_session_eval (the one-row lm_head).
- 32 sessions of the Qwen3-4B shape (1 layer) with prompts uniform in
  [64, 2048], then batched decode rounds: the benchmark's batch-32 decode
  (B = 32 GEMMs, split-KV attention over long unequal contexts).
- The Qwen3-14B heads (40 query / 8 KV heads, hidden 5120, FFN 17408; 1
  layer): a 2,048-token chunk after 10,240 prior positions, as the 14B
  chunked prefill reaches it.
- The prefill GEMMs at 2,048 token rows with the round's epilogues (store,
  residual add, SwiGLU of gate/up) and split-K 1, 2, 4 and the planner's.

One-layer models keep the oracle's work in seconds: with no logits wanted
the oracle stops a round after the last layer's K/V store (its append), so a
long prior context costs it only the K/V projections.  Rows the oracle
scores are a sample; every row the GPU computes takes the same path.
"""
import numpy as np
import pytest
import torch

import synthetic
from helpers import Pair, check_row, make_shape

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q3():
    import qwen3_dense_decoder_gb300 as q3
    q3.build()
    return q3


def _score_rows(T):
    return sorted(set(range(0, T, 64)) | {T - 1})


def test_qwen3_4b_one_2048_token_round():
    shape = make_shape("4b", n_layers=2)
    T = 2048
    pair = Pair(shape, seed=611, max_ctx=T + 64, max_round_tokens=T, n_blocks=2 * (T // 32 + 2),
                max_sessions=4)
    toks = synthetic.make_tokens(T, shape.vocab, seed=612)
    rows = _score_rows(T)
    g, o = pair.sessions(table=synthetic.make_block_permutation(pair.pool.n_blocks, seed=613)[:T // 32 + 1])
    lg = torch.empty(T, shape.vocab, dtype=torch.float32, device="cuda")
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    g.eval_n(torch.tensor(toks, device="cuda"), T, lg, am)
    pair.model.sync()
    ref = o.eval_rows(toks, rows)
    got = lg[rows].cpu().numpy()
    amx = am[rows].cpu().numpy()
    for i, r in enumerate(rows):
        c = check_row(got[i], ref[i], f"4b-2048/row{r}")
        assert c.ok, (r, c)
        assert amx[i] == c.argmax_gpu, r
    del lg
    # the benchmark's own call: q3_session_eval, the last row through the one-row lm_head
    g2 = pair.pool.session()
    g2.eval(torch.tensor(toks, device="cuda"), pair.logits[0], pair.amax[0:1])
    pair.model.sync()
    c = check_row(pair.logits[0].cpu().numpy(), ref[-1], "4b-2048/eval")
    assert c.ok, c
    assert int(pair.amax[0].item()) == c.argmax_gpu
    g.close()
    g2.close()


def test_qwen3_4b_batch_32_decode_over_prompts_64_to_2048():
    shape = make_shape("4b", n_layers=1)
    B, steps = 32, 4
    lens = synthetic.make_prompt_lengths(B, 64, 2048, seed=11)
    blocks = sum((int(n) + steps + 31) // 32 for n in lens) + 8
    pair = Pair(shape, seed=621, max_ctx=2048 + 64, max_round_tokens=2048, n_blocks=blocks,
                max_sessions=B + 2)
    perm = synthetic.make_block_permutation(blocks, seed=622)
    gs, os_, used = [], [], 0
    for i, n in enumerate(lens):
        nb = (int(n) + steps + 31) // 32
        g, o = pair.sessions(table=perm[used:used + nb])
        used += nb
        toks = synthetic.make_tokens(int(n), shape.vocab, seed=700 + i)
        g.eval(torch.tensor(toks, device="cuda"), pair.logits[0])
        o.append(toks)
        gs.append(g)
        os_.append(o)
    pair.model.sync()
    nxt = [[int(t)] for t in synthetic.make_tokens(B, shape.vocab, seed=623)]   # teacher-forced
    for step in range(steps):
        got, ref, am = pair.eval_batch(gs, os_, nxt)
        for i in range(B):
            c = check_row(got[i], ref[i], f"4b-b32/{int(lens[i])}")
            assert c.ok, (step, i, int(lens[i]), c)
            assert am[i] == c.argmax_gpu, (step, i)
        nxt = [[int(np.argmax(r))] for r in ref]
    for g in gs:
        g.close()


def test_qwen3_14b_heads_chunk_after_10240_positions():
    shape = make_shape("14b", n_layers=1)
    prior, T = 10240, 2048
    nb = (prior + T) // 32 + 2
    pair = Pair(shape, seed=631, max_ctx=prior + T + 64, max_round_tokens=T, n_blocks=nb + 8,
                max_sessions=2)
    g, o = pair.sessions(table=synthetic.make_block_permutation(nb + 8, seed=632)[:nb])
    toks = synthetic.make_tokens(prior + T, shape.vocab, seed=633)
    for a in range(0, prior, T):                     # the 14B workload's 2,048-token chunks
        g.eval(torch.tensor(toks[a:a + T], device="cuda"), pair.logits[0])
        o.append(toks[a:a + T])
    pair.model.sync()
    rows = _score_rows(T)
    lg = torch.empty(T, shape.vocab, dtype=torch.float32, device="cuda")
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    g.eval_n(torch.tensor(toks[prior:], device="cuda"), T, lg, am)
    pair.model.sync()
    ref = o.eval_rows(toks[prior:], rows)
    got = lg[rows].cpu().numpy()
    amx = am[rows].cpu().numpy()
    for i, r in enumerate(rows):
        c = check_row(got[i], ref[i], f"14b-late-chunk/row{r}")
        assert c.ok, (r, c)
        assert amx[i] == c.argmax_gpu, r
    g.close()


# ---------------------------------------------------------------- GEMM at 2,048 rows

def _w16(shape, seed, scale=0.05):
    g = torch.Generator(device="cuda").manual_seed(seed)
    # bf16-valued weights (exact in fp16), so the oracle's bf16 matmul takes them as they are
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


def _oracle_rows(orc, w, x, rows):
    wb = w.view(torch.int16).cpu().numpy().view(np.uint16)
    xs = x[rows].float().cpu().numpy()
    M, K = w.shape
    ref = orc.matmul(wb, 0, M, K, xs, n_threads=16).astype(np.float64)
    mag = np.abs(xs.astype(np.float64)) @ np.abs(w.float().cpu().numpy().astype(np.float64)).T
    return ref, mag


@pytest.mark.parametrize("M,K,epi,ks", [
    (6144, 2560, "store", 0),       # 4B QKV, planner's split
    (6144, 2560, "store", 2),
    (2560, 4096, "add", 2),         # 4B O + residual
    (2560, 9728, "add", 4),         # 4B down + residual
    (2560, 9728, "add", 0),
    (9728, 2560, "swiglu", 2),      # 4B gate/up + SwiGLU
    (9728, 2560, "swiglu", 0),
])
def test_prefill_gemm_epilogues_and_split_k_at_2048_rows(q3, orc, M, K, epi, ks):
    N = 2048
    rows = list(range(0, N, 32)) + [N - 1]
    x = torch.randn(N, K, generator=torch.Generator(device="cuda").manual_seed(M + K + ks),
                    device="cuda").to(torch.float16)
    w = _w16((M, K), 640 + ks)
    ref, mag = _oracle_rows(orc, w, x, rows)
    bound = 5e-5 * mag + 1e-30
    if epi == "swiglu":
        w2 = _w16((M, K), 650 + ks)
        ref_u, mag_u = _oracle_rows(orc, w2, x, rows)
        out = torch.empty(N, M, dtype=torch.float16, device="cuda")
        q3.op_gemm(w.to(torch.float16), x, N, q3.OP_SWIGLU, out, w2=w2.to(torch.float16), k_splits=ks)
        g, u = ref, ref_u
        sig = 1.0 / (1.0 + np.exp(-g))
        want = g * sig * u                                          # silu(g) * u
        dsilu = sig * (1.0 + g * (1.0 - sig))                       # |silu'| <= 1.1
        bnd = np.abs(dsilu) * 5e-5 * mag * np.abs(u) + np.abs(g * sig) * 5e-5 * mag_u
        bnd += 2.0 ** -11 * np.abs(want) + 2.0 ** -24              # fp16 output rounding
        gotv = out[rows].float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(gotv - want) <= bnd), (np.abs(gotv - want) / bnd).max()
        return
    init = torch.randn(N, M, generator=torch.Generator(device="cuda").manual_seed(7), device="cuda")
    out = init.clone() if epi == "add" else torch.empty(N, M, dtype=torch.float32, device="cuda")
    q3.op_gemm(w.to(torch.float16), x, N, q3.OP_ADD if epi == "add" else q3.OP_STORE, out, k_splits=ks)
    got = out[rows].cpu().numpy().astype(np.float64)
    if epi == "add":
        base = init[rows].cpu().numpy().astype(np.float64)
        want = base + ref
        bound = bound + 2.0 ** -23 * np.abs(want)                  # the FP32 residual add
    else:
        want = ref
    assert np.all(np.abs(got - want) <= bound), (np.abs(got - want) / bound).max()
