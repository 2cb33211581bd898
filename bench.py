#!/usr/bin/env python3
"""Benchmark of the GB300 forward on the Qwen3-4B shape.

Workload (seeded, synthetic, random-init weights of the shape): 36 layers,
hidden 2560, 32 query / 8 KV heads of width 128, FFN 9728, vocabulary
151,936, tied embedding, BF16 weights ~N(0, 0.02), paged BF16 KV in
32-position blocks.  A 2,048-token prompt is prefilled at batch 1, then the
session decodes greedily (the argmax of each step is the next token, on the
device).  Separately, 32 sessions with prompt lengths uniform in [64, 2048]
decode together.

A step is one decode token of the batch-1 session: one pass of every row of
the forward (embedding, RMSNorm, QKV, q/k norm + RoPE + KV append, paged GQA
attention, O, SwiGLU FFN, final norm, lm_head, argmax).  `value` is decode
tokens/s at batch 1 with inputs resident on the device; the weights (8 GB)
exceed L2, so no flush is needed between steps.  Prefill and batch-32 decode
are reported beside it.

Kernel rooflines come from a second, profiled pass of the same steps: the
library brackets every launch with CUDA events on its own stream
(q3_model_profile), and the dominant kernel's algorithmic bytes (or FLOPs)
per launch are divided by its mean launch time.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the forward has no cross-GPU exchange); value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Qwen3-4B-shape decode tok/s (% HBM roofline); prefill tok/s (% BF16 TC peak)"
# DRAM bytes read + written by one fused decode step over its algorithmic
# bytes, from ncu (dram__bytes_read.sum + dram__bytes_write.sum) on the
# 4-layer case; to be retaken whenever the kernel changes
DECODE_STEP_TRAFFIC_RATIO = (1.619629056e9 + 3.240704e6) / 1.6189e9
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256, help="timed decode steps")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--prompt", type=int, default=2048)
    ap.add_argument("--sessions", type=int, default=32)
    ap.add_argument("--no-b32", action="store_true", help="skip the batch-32 decode leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline leg")
    ap.add_argument("--shapes", nargs="*", default=None,
                    choices=("0.6b", "8b-q8_0", "14b", "4b-affine4", "14b-kvq8"),
                    help="measure the other named shapes instead (one JSON line each; 0.6b, 8b-q8_0 "
                         "and 14b if none given; 14b-kvq8 is the 14B workload over the Q8_0 K/V cache)")
    ap.add_argument("--ncu-case", choices=("decode-4layer", "gemm-gateup", "attn-prefill", "attn-decode-b32",
                                           "attn-decode-kvq8-b32", "gemv-a4", "prefill-2layer"),
                    default=None,
                    help="run only a small case sized for an ncu capture (a few GB on the device) and exit")
    return ap.parse_args()


def ncu_case(name: str):
    """Small cases for full ncu captures of the top kernels (the full-size
    workload holds ~20 GB and runs hundreds of launches)."""
    import torch

    import qwen3_dense_decoder_gb300 as q3
    import synthetic
    q3.build()
    if name == "decode-4layer":
        # the Qwen3-4B shape cut to 4 layers: a 2,048-token prefill, then fused
        # decode steps at context ~2,050 (about 1.6 GB streamed per step)
        s = synthetic.SHAPES["4b"].replace(n_layers=4)
        st = torch.cuda.Stream()
        torch.cuda.set_stream(st)
        w = synthetic.make_weights(s, seed=1234, device="cuda")
        m = q3.Model(s, w, max_ctx=2400, max_round_tokens=2048, stream=st)
        pool = m.pool(80, 2)
        ses = pool.session()
        lg = torch.empty(s.vocab, device="cuda")
        tok = torch.zeros(1, dtype=torch.int32, device="cuda")
        ses.eval(torch.tensor(synthetic.make_tokens(2048, s.vocab, 7), device="cuda"), lg, tok)
        for _ in range(6):
            ses.eval(tok, lg, tok)
        m.sync()
    elif name == "prefill-2layer":
        # one 2,048-token prefill round of the Qwen3-4B shape cut to 2 layers
        # (under 3 GB on the device): every prefill kernel once a layer, the
        # QKV GEMM with its head epilogue (q/k norm, RoPE, K/V append)
        s = synthetic.SHAPES["4b"].replace(n_layers=2)
        st = torch.cuda.Stream()
        torch.cuda.set_stream(st)
        w = synthetic.make_weights(s, seed=1234, device="cuda")
        m = q3.Model(s, w, max_ctx=2400, max_round_tokens=2048, stream=st)
        pool = m.pool(80, 2)
        ses = pool.session()
        lg = torch.empty(s.vocab, device="cuda")
        ses.eval(torch.tensor(synthetic.make_tokens(2048, s.vocab, 7), device="cuda"), lg)
        m.sync()
    elif name == "attn-decode-b32":
        # batch-32 decode of the Qwen3-4B shape cut to 2 layers: 32 sessions
        # with prompts U[64, 2048] (the bench's lengths), then 4 decode rounds
        s = synthetic.SHAPES["4b"].replace(n_layers=2)
        st = torch.cuda.Stream()
        torch.cuda.set_stream(st)
        w = synthetic.make_weights(s, seed=1234, device="cuda")
        B = 32
        m = q3.Model(s, w, max_ctx=2400, max_round_tokens=2048, stream=st)
        pool = m.pool(B * 75 + 8, B + 2)
        lg = torch.empty(B, s.vocab, device="cuda")
        am = torch.zeros(B, dtype=torch.int32, device="cuda")
        lens = synthetic.make_prompt_lengths(B, 64, 2048, seed=11)
        ss = [pool.session() for _ in range(B)]
        for i, x in enumerate(ss):
            x.eval(torch.tensor(synthetic.make_tokens(int(lens[i]), s.vocab, seed=100 + i), device="cuda"),
                   lg[0], am[i:i + 1])
        toks = am.clone()
        for _ in range(4):
            m.eval_batch(ss, toks, [1] * B, lg, toks)
        m.sync()
    elif name == "attn-decode-kvq8-b32":
        # the same batch-32 decode over the opt-in Q8_0 K/V cache
        s = synthetic.SHAPES["4b"].replace(n_layers=2, kv_quant=synthetic.Q8_0)
        st = torch.cuda.Stream()
        torch.cuda.set_stream(st)
        w = synthetic.make_weights(s, seed=1234, device="cuda")
        B = 32
        m = q3.Model(s, w, max_ctx=2400, max_round_tokens=2048, stream=st)
        pool = m.pool(B * 75 + 8, B + 2)
        lg = torch.empty(B, s.vocab, device="cuda")
        am = torch.zeros(B, dtype=torch.int32, device="cuda")
        lens = synthetic.make_prompt_lengths(B, 64, 2048, seed=11)
        ss = [pool.session() for _ in range(B)]
        for i, x in enumerate(ss):
            x.eval(torch.tensor(synthetic.make_tokens(int(lens[i]), s.vocab, seed=100 + i), device="cuda"),
                   lg[0], am[i:i + 1])
        toks = am.clone()
        for _ in range(4):
            m.eval_batch(ss, toks, [1] * B, lg, toks)
        m.sync()
    elif name == "gemv-a4":
        # the gate/up projection of a Qwen3-4B AFFINE4_GS32 decode step as one
        # operator call: 19,456 x 2,560 weights, 31 MB at 5.0 bits a weight
        M, K = 19456, 2560
        g = torch.Generator(device="cuda")
        g.manual_seed(8)
        w = (torch.randn(M, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        groups = q3.quantize_affine4(w)
        x = torch.randn(K, device="cuda", generator=g)
        for _ in range(6):
            q3.op_matvec_affine4(groups, x, M, K)
        torch.cuda.synchronize()
    elif name == "attn-prefill":
        # one layer's prefill attention of a 2,048-token round of the Qwen3-4B
        # shape (32 query / 8 KV heads) over a permuted block table
        T, n_q, n_kv = 2048, 32, 8
        nblk = T // 32
        g = torch.Generator(device="cuda")
        g.manual_seed(6)
        q = torch.randn(T, n_q, 128, device="cuda", generator=g).to(torch.float16)
        kv = torch.randn(nblk + 8, 2, n_kv, 32, 128, device="cuda", generator=g).to(torch.bfloat16)
        table = torch.from_numpy(synthetic.make_block_permutation(nblk + 8, seed=7)[:nblk]).cuda()
        for _ in range(6):
            q3.op_prefill_attention(q, kv, table, 0, n_kv)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(True), torch.cuda.Event(True)
        a.record()
        for _ in range(10):
            q3.op_prefill_attention(q, kv, table, 0, n_kv)
        b.record()
        b.synchronize()
        us = a.elapsed_time(b) / 10 * 1e3
        fl = 4.0 * 128 * n_q * T * (T + 1) / 2
        print(f"prefill attention T={T}: {us:.1f} us/call (with its metadata upload and sync), "
              f"{fl / us / 1e6:.1f} TFLOP/s", flush=True)
    else:
        # the gate/up projection of a 2,048-token prefill of the Qwen3-4B shape
        M, N, K = 19456, 2048, 2560
        g = torch.Generator(device="cuda")
        g.manual_seed(5)
        w = (torch.randn(M, K, device="cuda", generator=g) * 0.02).to(torch.float16)
        x = torch.randn((N + 255) // 256 * 256, K, device="cuda", generator=g).to(torch.float16)
        for _ in range(6):
            q3.op_matmul(w, x, N)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(True), torch.cuda.Event(True)
        a.record()
        for _ in range(10):
            q3.op_matmul(w, x, N)
        b.record()
        b.synchronize()
        us = a.elapsed_time(b) / 10 * 1e3
        print(f"gemm {M}x{N}x{K}: {us:.1f} us/launch, {2.0 * M * N * K / us / 1e6:.1f} TFLOP/s", flush=True)
    print("ok", name, flush=True)


# ---------------------------------------------------------------- algorithmic work

def proj_params(s) -> int:
    per_layer = (s.q_width + 2 * s.kv_width) * s.hidden + s.hidden * s.q_width + 3 * s.ffn * s.hidden
    return per_layer * s.n_layers


def decode_bytes(s, ctx: int, batch: int = 1, ctxs=None) -> float:
    """HBM bytes one decode step must move: every weight once (bf16) plus the
    K and V of every cached position of every session, per layer."""
    w = 2.0 * proj_params(s) + 2.0 * s.vocab * s.hidden
    kv_per_pos = s.n_layers * 2 * s.kv_width * 2
    total_ctx = sum(ctxs) if ctxs is not None else ctx * batch
    return w + kv_per_pos * total_ctx


def prefill_flops(s, T: int) -> float:
    """2 * params * tokens for the projections, causal attention (QK^T and PV
    over T^2/2 pairs), and the lm_head of the last row."""
    return (2.0 * proj_params(s) * T + 2.0 * s.n_layers * s.q_width * T * T
            + 2.0 * s.vocab * s.hidden)


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi samples every 200 ms while a timed region runs."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        return clock_summary(getattr(self, "lines", []))


def clock_summary(lines) -> dict:
    """Median SM clock, the largest max clock and the throttle reasons seen
    in nvidia-smi sample lines (the CLOCK_FIELDS columns)."""
    if True:
        mhz, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(mhz)}


# ---------------------------------------------------------------- GPU arm

class Timer:
    """CUDA events on the library's stream."""

    def __init__(self, stream):
        import torch
        self.stream = stream
        self.a = torch.cuda.Event(enable_timing=True)
        self.b = torch.cuda.Event(enable_timing=True)

    def start(self):
        self.a.record(self.stream)

    def stop(self) -> float:
        self.b.record(self.stream)
        self.b.synchronize()
        return self.a.elapsed_time(self.b)


def barrier(dist_on: bool):
    if dist_on:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, dist_on: bool) -> float:
    if not dist_on:
        return v
    import torch
    import torch.distributed as dist
    # NCCL reduces device tensors; gloo (CPU tests of this path) host tensors
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def decode_loop(sess, tok, logits, steps: int):
    """steps greedy decode steps at batch 1: each step's argmax is written over
    its own input token, so the next step reads it on the device."""
    for _ in range(steps):
        sess.eval(tok, logits, tok)


def run_gpu(args, dist_on: bool, rank: int, world: int):
    import numpy as np
    import torch

    import qwen3_dense_decoder_gb300 as q3
    import synthetic

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    q3.build()
    shape = synthetic.SHAPES["4b"]
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    W, K, P = args.warmup, args.steps, args.prompt
    max_ctx = P + W + 4 * K + 64      # value, profiled, per-operation and e2e passes share the session
    w = synthetic.make_weights(shape, seed=1234, device="cuda")
    model = q3.Model(shape, w, max_ctx=max_ctx, max_round_tokens=P, stream=stream)
    n_sess = 2 + (0 if args.no_b32 else args.sessions)     # decode + profiled-prefill sessions
    blocks_per = (max_ctx + 31) // 32
    pool = model.pool(n_blocks=blocks_per * n_sess + 8, max_sessions=n_sess + 2)
    V = shape.vocab
    logits = torch.empty(max(args.sessions, 1), V, dtype=torch.float32, device="cuda")
    amax = torch.empty(max(args.sessions, 1), dtype=torch.int32, device="cuda")
    timer = Timer(stream)
    out = {}

    # ---- prefill at batch 1: a 2,048-token prompt into an empty session
    prompt = torch.tensor(synthetic.make_tokens(P, V, seed=7), device="cuda")
    sess = pool.session()
    pre_ms = []
    for it in range(W + 3):
        sess.reset()
        torch.cuda.synchronize()
        timer.start()
        sess.eval(prompt, logits[0], amax[0:1])
        ms = timer.stop()
        if it >= W:
            pre_ms.append(ms)
    model.sync()
    out["prefill_ms"] = statistics.median(pre_ms)

    # ---- decode at batch 1 (the value): W warm-up steps, then K timed steps
    tok = amax[0:1].clone()
    decode_loop(sess, tok, logits[0], W)
    model.sync()
    ctx0 = sess.pos
    barrier(dist_on)
    torch.cuda.synchronize()
    l0 = model.launch_count
    with ClockSampler(local) as clk:
        timer.start()
        decode_loop(sess, tok, logits[0], K)
        dec_ms = timer.stop()
    torch.cuda.synchronize()
    barrier(dist_on)
    model.sync()
    out["launches"] = model.launch_count - l0
    out["decode_ms"] = dec_ms
    out["decode_ctx"] = (ctx0 + 1, ctx0 + K)
    out["clocks"] = clk.summary()

    # ---- profiled pass of the same decode steps (per-kernel CUDA events)
    p0 = sess.pos
    model.profile(True)
    model.profile_reset()
    decode_loop(sess, tok, logits[0], K)
    out["decode_profile"] = model.profile_read()
    out["decode_profile_ctx"] = (p0 + 1, p0 + K)
    model.profile(False)
    # ---- the same decode steps on the per-operation path (one launch per
    # operation), for comparison with the fused step
    out["fused"] = model.fused_decode
    if model.fused_decode:
        model.set_fused_decode(False)
        decode_loop(sess, tok, logits[0], 2)
        model.sync()
        q0 = sess.pos
        timer.start()
        decode_loop(sess, tok, logits[0], K)
        out["per_op_ms"] = timer.stop()
        out["per_op_ctx"] = (q0 + 1, q0 + K)
        model.set_fused_decode(True)
        model.sync()
    # ---- profiled prefill
    sess2 = pool.session()
    model.profile(True)
    model.profile_reset()
    sess2.eval(prompt, logits[0], amax[0:1])
    out["prefill_profile"] = model.profile_read()
    model.profile(False)
    sess2.close()

    # ---- end to end through the C ABI with host buffers: per step the token
    # goes host->device from pinned memory and the logits and argmax come back
    h_tok = torch.empty(1, dtype=torch.int32, pin_memory=True)
    h_logits = torch.empty(V, dtype=torch.float32, pin_memory=True)
    h_am = torch.empty(1, dtype=torch.int32, pin_memory=True)
    h_tok.copy_(tok.cpu())
    d_tok = torch.empty(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(K):
        d_tok.copy_(h_tok, non_blocking=True)
        sess.eval(d_tok, logits[0], amax[0:1])
        h_logits.copy_(logits[0], non_blocking=True)
        h_am.copy_(amax[0:1], non_blocking=True)
        stream.synchronize()
        h_tok.copy_(h_am)
    e2e_s = time.perf_counter() - t0
    model.sync()
    out["e2e_s"] = e2e_s
    out["e2e_bytes"] = (4, 4 * V + 4)
    sess.close()

    # ---- decode at 32 sessions, prompts uniform in [64, 2048]
    if not args.no_b32:
        B = args.sessions
        lens = synthetic.make_prompt_lengths(B, 64, P, seed=11)
        sessions = [pool.session() for _ in range(B)]
        for i, s in enumerate(sessions):
            s.eval(torch.tensor(synthetic.make_tokens(int(lens[i]), V, seed=100 + i), device="cuda"),
                   logits[0], amax[i:i + 1])
        model.sync()
        toks = amax[:B].clone()
        ones = [1] * B
        for _ in range(W):
            model.eval_batch(sessions, toks, ones, logits[:B], toks)
        model.sync()
        ctx_b = [s.pos for s in sessions]
        barrier(dist_on)
        torch.cuda.synchronize()
        with ClockSampler(local) as clk_b32:
            timer.start()
            for _ in range(K):
                model.eval_batch(sessions, toks, ones, logits[:B], toks)
            b32_ms = timer.stop()
        out["b32_clocks"] = clk_b32.summary()
        model.sync()
        model.profile(True)
        model.profile_reset()
        for _ in range(min(K, 32)):
            model.eval_batch(sessions, toks, ones, logits[:B], toks)
        out["b32_profile"] = model.profile_read()
        out["b32_profile_steps"] = min(K, 32)
        model.profile(False)
        out["b32_ms"] = b32_ms
        out["b32_ctx"] = [c + K / 2 for c in ctx_b]
        for s in sessions:
            s.close()
    out["shape"] = shape
    out["weights"] = w
    return out


# ---------------------------------------------------------------- CPU baseline (the oracle)

def oracle_decode_sample(shape, weights, budget_s: float, max_steps: int, warmup: int = 1):
    """Time the oracle (plain C, FP64 accumulation) on greedy decode steps of
    the same shape after a 16-token prompt, on this host's cores."""
    import numpy as np

    import oracle
    import synthetic
    oracle.build()
    m = oracle.Model(shape, weights)
    s = m.session(max_ctx=16 + warmup + max_steps + 1)
    lg = s.eval(synthetic.make_tokens(16, shape.vocab, seed=7))
    tok = int(np.argmax(lg))
    for _ in range(warmup):
        tok = int(np.argmax(s.eval([tok])))
    t0 = time.perf_counter()
    steps = 0
    while steps < max_steps:
        tok = int(np.argmax(s.eval([tok])))
        steps += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    ctx = 16 + warmup
    return {"value": steps / dt, "unit": "tok/s", "cores": m.n_threads, "kind": "oracle",
            "sample": (f"{steps} greedy decode steps of the full {shape.n_layers}-layer {shape.name} shape "
                       f"at batch 1 after a 16-token prompt (context {ctx + 1}..{ctx + steps}; at that "
                       f"length attention is a few percent of a step's work)"),
            "seconds": dt, "steps": steps}


def oracle_prefill_sample(shape, weights, tokens: int) -> dict:
    """Time the oracle on one prefill round of `tokens` seeded tokens of the
    full-depth shape (logits of the last row), on this host's cores."""
    import oracle
    import synthetic
    oracle.build()
    m = oracle.Model(shape, weights)
    s = m.session(max_ctx=tokens + 1)
    toks = synthetic.make_tokens(tokens, shape.vocab, seed=7)
    t0 = time.perf_counter()
    s.eval(toks)
    dt = time.perf_counter() - t0
    return {"value": round(tokens / dt, 3), "unit": "tok/s", "cores": m.n_threads, "seconds": round(dt, 2),
            "sample": f"one {tokens}-token prefill round of the full {shape.n_layers}-layer {shape.name} shape"}


# ---------------------------------------------------------------- other named shapes

def q8_bytes(params: int) -> float:
    """Q8_0 bytes of `params` weights: 34-byte blocks of 32."""
    return params * 34.0 / 32.0


def affine4_bytes(params: int) -> float:
    """AFFINE4_GS32 bytes of `params` weights: 20-byte groups of 32 (5.0 bits a weight)."""
    return params * 20.0 / 32.0


def step_bytes(s, ctxs) -> float:
    """HBM bytes of one decode step: every projection once (bf16, Q8_0 blocks
    or AFFINE4 groups: the format's bytes, whatever copy the kernels read), the
    lm_head once (bf16), and the K/V of every cached position of every session
    (2 bytes a value in BF16, 34 bytes per 32 values with the Q8_0 cache)."""
    p = proj_params(s)
    pw = {1: q8_bytes(p), 2: affine4_bytes(p)}.get(s.scheme, 2.0 * p)
    w = pw + 2.0 * s.vocab * s.hidden
    kv_b = 34.0 / 32.0 if getattr(s, "kv_quant", 0) == 1 else 2.0
    return w + s.n_layers * 2 * s.kv_width * kv_b * float(sum(ctxs))


def run_shape(name: str, pk: dict, pk_kind: str, with_oracle: bool) -> dict:
    """The named workload of one shape ("Kipp Model Support", section "The
    registry"): 0.6B -- a 128-token prompt, 64 greedy decode steps, and a ragged
    3-round prefill (5, 40, 83); 8B Q8_0 -- a 2,048-token prefill, then decode at
    batch 1 and at 32 sessions with prompts U[64, 2048] (the same for 4B
    AFFINE4_GS32, the scheme of "Kipp Roadmap", status v0.0.4's 2,048-token
    prefill figures); 14B -- a 12,800-token
    prefill in 2,048-token chunks, then 8 sessions decoding 128 tokens at a
    16,384-token context over one shared block pool with permuted tables
    (14b-kvq8: the same over the opt-in Q8_0 K/V cache)."""
    import numpy as np
    import torch

    import qwen3_dense_decoder_gb300 as q3
    import synthetic
    s = synthetic.SHAPES["14b"].replace(kv_quant=synthetic.Q8_0, name="qwen3-14b-kv-q8_0") \
        if name == "14b-kvq8" else synthetic.SHAPES[name]
    st = torch.cuda.Stream()
    torch.cuda.set_stream(st)
    w = synthetic.make_weights(s, seed=1234, device="cuda")     # bf16 source (the oracle packs its own)
    wg = w
    if s.scheme in (synthetic.Q8_0, synthetic.AFFINE4):
        pack = q3.quantize_q8_0 if s.scheme == synthetic.Q8_0 else q3.quantize_affine4
        wg = dict(w, layers=[dict(lw) for lw in w["layers"]])
        for lw in wg["layers"]:
            for nm in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
                lw[nm] = pack(lw[nm])
    V = s.vocab

    clock_lines = []      # nvidia-smi samples taken during every timed region of the shape

    def timed(fn):
        a, b = torch.cuda.Event(True), torch.cuda.Event(True)
        torch.cuda.synchronize()
        with ClockSampler(torch.cuda.current_device()) as clk:
            a.record(st)
            fn()
            b.record(st)
            b.synchronize()
        clock_lines.extend(clk.lines)
        return a.elapsed_time(b)

    dtype = {synthetic.BF16: "bf16", synthetic.Q8_0: "q8_0 weights, fp16/bf16 compute",
             synthetic.AFFINE4: "affine4_gs32 weights, fp16/bf16 compute"}[s.scheme]
    if getattr(s, "kv_quant", synthetic.BF16) == synthetic.Q8_0:
        dtype += "; q8_0 K/V cache"
    out = {"shape": s.name, "n_gpus": 1, "dtype": dtype,
           "data": "synthetic (seeded random-init weights and tokens)", "peak_kind": pk_kind}
    lg = torch.empty(max(32, 8), V, dtype=torch.float32, device="cuda")
    am = torch.zeros(max(32, 8), dtype=torch.int32, device="cuda")
    peak_tf, peak_gb = pk["bf16_tflops"], pk["hbm_gbs"]

    def prefill_entry(T, ms, flops=None):
        fl = flops if flops is not None else prefill_flops(s, T)
        return {"tokens": T, "ms": round(ms, 3), "tok_s": round(T / ms * 1e3, 1),
                "tflops": round(fl / ms / 1e9, 1), "tc_frac": round(fl / ms / 1e9 / peak_tf, 4)}

    def decode_entry(sessions, steps, ms, ctxs):
        by = step_bytes(s, ctxs)
        return {"sessions": sessions, "steps": steps, "ms_per_step": round(ms / steps, 4),
                "tok_s": round(sessions * steps / ms * 1e3, 1), "bytes_per_step": by,
                "hbm_frac": round(by / (ms / steps) / 1e6 / peak_gb, 4)}

    if name == "0.6b":
        m = q3.Model(s, wg, max_ctx=512, max_round_tokens=2048, stream=st)
        pool = m.pool(16, 2)
        ses = pool.session()
        toks = torch.tensor(synthetic.make_tokens(128, V, seed=7), device="cuda")
        pre = []
        for i in range(4):
            ses.reset()
            t = timed(lambda: ses.eval(toks, lg[0], am[0:1]))
            if i:
                pre.append(t)
        out["prefill_128"] = prefill_entry(128, statistics.median(pre))
        tok = am[0:1].clone()
        for _ in range(3):
            ses.eval(tok, lg[0], tok)
        c0 = ses.pos
        ms = timed(lambda: [ses.eval(tok, lg[0], tok) for _ in range(64)])
        out["decode_b1"] = decode_entry(1, 64, ms, [c0 + 32])
        ses.reset()
        rounds = [5, 40, 83]
        rt = torch.tensor(synthetic.make_tokens(sum(rounds), V, seed=8), device="cuda")

        def ragged():
            a = 0
            for n in rounds:
                ses.eval(rt[a:a + n], lg[0], am[0:1])
                a += n
        ragged()
        ses.reset()
        ms = timed(ragged)
        out["prefill_ragged_5_40_83"] = prefill_entry(sum(rounds), ms)
        ses.close()
    elif name in ("8b-q8_0", "4b-affine4"):
        m = q3.Model(s, wg, max_ctx=2400, max_round_tokens=2048, stream=st)
        pool = m.pool(34 * 75 + 8, 36)
        ses = pool.session()
        toks = torch.tensor(synthetic.make_tokens(2048, V, seed=7), device="cuda")
        pre = []
        for i in range(3):
            ses.reset()
            t = timed(lambda: ses.eval(toks, lg[0], am[0:1]))
            if i:
                pre.append(t)
        out["prefill_2048"] = prefill_entry(2048, statistics.median(pre))
        tok = am[0:1].clone()
        for _ in range(3):
            ses.eval(tok, lg[0], tok)
        c0 = ses.pos
        ms = timed(lambda: [ses.eval(tok, lg[0], tok) for _ in range(64)])
        out["decode_b1"] = decode_entry(1, 64, ms, [c0 + 32])
        ses.close()
        B = 32
        lens = synthetic.make_prompt_lengths(B, 64, 2048, seed=11)
        ss = [pool.session() for _ in range(B)]
        for i, x in enumerate(ss):
            x.eval(torch.tensor(synthetic.make_tokens(int(lens[i]), V, seed=100 + i), device="cuda"),
                   lg[0], am[i:i + 1])
        bt = am[:B].clone()
        for _ in range(3):
            m.eval_batch(ss, bt, [1] * B, lg[:B], bt)
        ctxs = [x.pos + 8 for x in ss]
        ms = timed(lambda: [m.eval_batch(ss, bt, [1] * B, lg[:B], bt) for _ in range(16)])
        out["decode_b32"] = decode_entry(B, 16, ms, ctxs)
        for x in ss:
            x.close()
    else:
        B, CTX, STEPS, CHUNK = 8, 16384, 128, 2048
        nblk = (CTX + STEPS + 31) // 32
        m = q3.Model(s, wg, max_ctx=CTX + STEPS + 64, max_round_tokens=CHUNK, stream=st)
        pool = m.pool(B * nblk + 16, B + 1)
        perm = synthetic.make_block_permutation(B * nblk + 16, seed=21)
        ss = []
        for i in range(B):
            x = pool.session()
            x.set_block_table(perm[i * nblk:(i + 1) * nblk])
            ss.append(x)
        toks = torch.tensor(synthetic.make_tokens(CTX, V, seed=9), device="cuda")

        def chunks(x, lo, hi):
            for a in range(lo, hi, CHUNK):
                x.eval(toks[a:min(hi, a + CHUNK)], lg[0], am[0:1])
        ms = timed(lambda: chunks(ss[0], 0, 12800))
        fl = 2.0 * proj_params(s) * 12800 + 2.0 * s.n_layers * s.q_width * 12800 * 12800 \
            + 2.0 * V * s.hidden * ((12800 + CHUNK - 1) // CHUNK)
        out["prefill_12800_chunked"] = prefill_entry(12800, ms, fl)
        chunks(ss[0], 12800, CTX)
        for x in ss[1:]:
            chunks(x, 0, CTX)
        bt = am[:B].clone()
        for _ in range(2):
            m.eval_batch(ss, bt, [1] * B, lg[:B], bt)
        ctxs = [x.pos + STEPS // 2 for x in ss]
        ms = timed(lambda: [m.eval_batch(ss, bt, [1] * B, lg[:B], bt) for _ in range(STEPS)])
        out["decode_8x16k"] = decode_entry(B, STEPS, ms, ctxs)
        for x in ss:
            x.close()
    m.sync()
    out["clocks"] = clock_summary(clock_lines)
    out["gpu_launches_total"] = m.launch_count
    del m
    torch.cuda.synchronize()
    if with_oracle:
        cb = oracle_decode_sample(s, w, budget_s=8.0, max_steps=8)
        cb.pop("steps", None)
        cb.pop("seconds", None)
        out["cpu_baseline"] = cb
    del w, wg
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- report

def workload_config(args):
    return {"workload": (f"qwen3-4b-shape (36 layers, hidden 2560, 32/8 heads x 128, FFN 9728, "
                         f"vocab 151936, tied, bf16 N(0,0.02) random init); {args.prompt}-token "
                         f"prefill at batch 1, then {args.steps} greedy decode steps at batch 1 "
                         f"(value) and at {args.sessions} sessions with prompts U[64, {args.prompt}]"),
            "l2": "inputs larger than L2: 8.0 GB of weights streamed per decode step",
            "kv": "paged bf16, 32-position blocks", "parallelism": f"replicas x{args.gpus}"}


def report(args, res, world, dist_on, pk, pk_kind):
    s = res["shape"]
    K = args.steps
    dec_ms = max_over_ranks(res["decode_ms"], dist_on)
    value = world * K / (dec_ms / 1e3)
    c0, c1 = res["decode_ctx"]
    mean_ctx = (c0 + c1) / 2
    step_bytes = decode_bytes(s, mean_ctx)
    w_bytes = 2.0 * proj_params(s) + 2.0 * s.vocab * s.hidden
    prof = res["decode_profile"]
    if prof.get("decode_step", (0, 0))[1]:
        # the fused step: one launch streams every weight and the KV context
        k_ms, k_n = prof["decode_step"]
        pc0, pc1 = res["decode_profile_ctx"]
        k_bytes = decode_bytes(s, (pc0 + pc1) / 2)
        k_name = "decode_step (fused one-kernel decode step: all projections, attention, lm_head)"
        # DRAM bytes of one launch from an ncu capture of the 4-layer case
        # (bench.py --ncu-case decode-4layer): 1.0025 x its algorithmic bytes,
        # scaled to this launch by the same ratio
        k_traffic = round(DECODE_STEP_TRAFFIC_RATIO * k_bytes)
    else:
        k_ms, k_n = prof["gemv"]
        k_bytes = w_bytes * K / k_n
        k_name = "gemv (decode matvec, all projections + lm_head)"
        k_traffic = None
    k_achieved = k_bytes / (k_ms / k_n / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(dec_ms / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random-init weights and tokens of the named shape)",
        "config": workload_config(args),
        "hbm_roofline": {"achieved_gbs": round(step_bytes * value / world / 1e9, 1),
                         "bytes_per_step": step_bytes, "peak_gbs": pk["hbm_gbs"],
                         "frac": round(step_bytes * value / world / 1e9 / pk["hbm_gbs"], 4),
                         "peak_kind": pk_kind},
        "roofline": {"kernel": k_name, "bound": "hbm",
                     "achieved": round(k_achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(k_achieved / pk["hbm_gbs"], 4), "traffic": k_traffic,
                     "bytes_per_launch": k_bytes, "launches": k_n,
                     "mean_launch_us": round(k_ms / k_n * 1e3, 3), "peak_kind": pk_kind},
        "clocks": res["clocks"],
        "gpu_launches": res["launches"],
        "decode_kernels_ms_per_step": {k: round(v[0] / K, 4) for k, v in res["decode_profile"].items()},
    }
    if "per_op_ms" in res:
        q0, q1 = res["per_op_ctx"]
        po_ms = max_over_ranks(res["per_op_ms"], dist_on)
        line["decode_per_op_path"] = {
            "value": round(world * K / (po_ms / 1e3), 2), "unit": "tok/s", "ms_per_step": round(po_ms / K, 4),
            "hbm_frac": round(decode_bytes(s, (q0 + q1) / 2) * K / (po_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
            "note": "same steps, one launch per operation (q3_model_set_fused_decode(m, 0))"}
    # prefill
    P = args.prompt
    pre_ms = max_over_ranks(res["prefill_ms"], dist_on)
    fl = prefill_flops(s, P)
    gemm_ms, gemm_n = res["prefill_profile"]["gemm"]
    gemm_fl = 2.0 * proj_params(s) * P
    line["prefill"] = {
        "value": round(world * P / (pre_ms / 1e3), 1), "unit": "tok/s", "ms": round(pre_ms, 3),
        "tc_roofline": {"achieved_tflops": round(fl / (pre_ms / 1e3) / 1e12, 1),
                        "peak": pk["bf16_tflops"], "frac": round(fl / (pre_ms / 1e3) / 1e12 / pk["bf16_tflops"], 4),
                        "flops": fl, "peak_kind": pk_kind},
        "roofline": {"kernel": "gemm (tcgen05 projections)", "bound": "tensor",
                     "achieved": round(gemm_fl / (gemm_ms / 1e3) / 1e12, 1), "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(gemm_fl / (gemm_ms / 1e3) / 1e12 / pk["bf16_tflops"], 4),
                     "traffic": None, "launches": gemm_n, "peak_kind": pk_kind},
        "kernels_ms": {k: round(v[0], 3) for k, v in res["prefill_profile"].items()},
    }
    if "b32_ms" in res:
        B = args.sessions
        b_ms = max_over_ranks(res["b32_ms"], dist_on)
        b_val = world * B * K / (b_ms / 1e3)
        b_bytes = decode_bytes(s, 0, ctxs=res["b32_ctx"])
        line["decode_b32"] = {
            "value": round(b_val, 1), "unit": "tok/s", "ms_per_step": round(b_ms / K, 4),
            "hbm_roofline": {"achieved_gbs": round(b_bytes * K / (b_ms / 1e3) / 1e9, 1),
                             "bytes_per_step": b_bytes,
                             "frac": round(b_bytes * K / (b_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)},
            "kernels_ms_per_step": {k: round(v[0] / res["b32_profile_steps"], 4)
                                    for k, v in res["b32_profile"].items()},
            "clocks": res["b32_clocks"],
        }
    e_s = max_over_ranks(res["e2e_s"], dist_on)
    line["e2e"] = {"value": round(world * K / e_s, 2), "unit": "tok/s",
                   "h2d_bytes_per_step": res["e2e_bytes"][0], "d2h_bytes_per_step": res["e2e_bytes"][1]}
    return line


# ---------------------------------------------------------------- main

def reference_arm(args, rank: int):
    """The oracle timed on this host's cores, on the same metric and workload shape."""
    if rank != 0:
        return
    import synthetic
    shape = synthetic.SHAPES["4b"]
    w = synthetic.make_weights(shape, seed=1234, device="cpu")
    # every timed step is one full decode token; the count is capped so the
    # run stays within a few minutes
    cb = oracle_decode_sample(shape, w, budget_s=120.0, max_steps=args.steps, warmup=args.warmup)
    line = {"metric": METRIC, "value": round(cb["value"], 4), "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 / cb["value"], 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded random-init weights and tokens of the named shape)",
            "config": workload_config(args), "impl": "reference",
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": round(cb["value"], 4), "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    line["cpu_baseline"]["sample"] += f"; {cb['steps']} of the {args.steps} requested steps timed"
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.ncu_case:
        ncu_case(args.ncu_case)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist_on = world > 1
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if dist_on:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    pk, pk_kind = peaks()
    if args.shapes is not None:
        for name in args.shapes or ["0.6b", "8b-q8_0", "14b"]:
            if rank == 0:
                print(json.dumps(run_shape(name, pk, pk_kind, with_oracle=not args.no_cpu)), flush=True)
        return
    res = run_gpu(args, dist_on, rank, world)
    line = report(args, res, world, dist_on, pk, pk_kind)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = oracle_decode_sample(res["shape"], res["weights"], budget_s=20.0,
                                                    max_steps=16)
        for k in ("seconds", "steps"):
            line["cpu_baseline"].pop(k, None)
        # the oracle's prefill beside the GPU's (a bounded sample: one 64-token round)
        line["cpu_baseline"]["prefill"] = oracle_prefill_sample(res["shape"], res["weights"], 64)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist_on:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
