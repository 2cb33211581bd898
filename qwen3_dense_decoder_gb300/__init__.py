"""Python binding of libq3.so, the sm_103a forward of a dense Qwen3-style decoder.

The binding only marshals arguments: every step of the forward runs in the
library's CUDA kernels (include/q3.h documents each entry point).  PyTorch is
used for device memory and streams.  There is no fallback: if the library is
missing or the device is not an sm_103 GPU, the calls raise.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libq3.so")

BF16, Q8_0, AFFINE4 = 0, 1, 2
KV_BLOCK = 32
Q8_0_BYTES = 34
AFFINE4_BYTES = 20
ERRORS = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED_DEVICE", -3: "OOM", -4: "POOL_EXHAUSTED",
          -5: "CTX_OVERFLOW", -6: "CUDA", -7: "DEVICE_CHECK", -8: "POISONED"}

PROJ = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


class Q3Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class _Config(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("hidden", C.c_int), ("n_q_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("max_ctx", C.c_int), ("rope_theta", C.c_float),
                ("rms_eps", C.c_float), ("tied", C.c_int), ("scheme", C.c_int),
                ("kv_scheme", C.c_int)]


class _LayerW(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
                                         "ffn_norm", "w_gate", "w_up", "w_down")]


class _Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", C.c_void_p),
                ("layers", C.POINTER(_LayerW))]


_lib = None


def build(force: bool = False) -> str:
    from . import buildlib
    return buildlib.build(force=force)


def lib():
    """The loaded libq3.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "qwen3_dense_decoder_gb300.build() (nvcc, sm_103a)")
        L = C.CDLL(LIB_PATH)
        vp, i, i64 = C.c_void_p, C.c_int, C.c_int64
        L.q3_last_error.restype = C.c_char_p
        L.q3_model_create.argtypes = [C.POINTER(_Config), C.POINTER(_Weights), i, vp, C.POINTER(vp)]
        L.q3_model_destroy.argtypes = [vp]
        L.q3_pool_create.argtypes = [vp, i, i, C.POINTER(vp)]
        L.q3_pool_destroy.argtypes = [vp]
        L.q3_session_create.argtypes = [vp, C.POINTER(vp)]
        L.q3_session_destroy.argtypes = [vp]
        L.q3_session_set_block_table.argtypes = [vp, vp, i]
        L.q3_session_eval.argtypes = [vp, vp, i, vp, vp]
        L.q3_eval_batch.argtypes = [vp, i, vp, vp, vp, vp]
        L.q3_session_truncate.argtypes = [vp, i]
        L.q3_pool_enable_prefix.argtypes = [vp, i]
        L.q3_session_publish.argtypes = [vp, vp, i, vp]
        L.q3_session_attach_prefix.argtypes = [vp, vp, i, vp]
        L.q3_session_reset.argtypes = [vp]
        L.q3_session_pos.argtypes = [vp]
        L.q3_sync.argtypes = [vp]
        L.q3_quantize_q8_0.argtypes = [vp, i64, vp, vp]
        L.q3_quantize_affine4.argtypes = [vp, i64, vp, vp]
        L.q3_affine4_to_f16.argtypes = [vp, i64, vp, vp]
        L.q3_model_launch_count.argtypes = [vp]
        L.q3_model_launch_count.restype = i64
        L.q3_op_matmul.argtypes = [vp, vp, i, i, i, vp, i, vp]
        L.q3_op_matmul_splitk_noalloc.argtypes = [vp, vp, i, i, i, i, vp, vp]
        L.q3_op_gemm.argtypes = [vp, vp, vp, i, i, i, i, vp, i, i, vp]
        L.q3_gemm_plan.argtypes = [i, i, i, C.POINTER(i), C.POINTER(i)]
        L.q3_attention_plan.argtypes = [i, i, i, C.POINTER(i)]
        L.q3_noalloc_last_error.restype = C.c_char_p
        L.q3_model_profile.argtypes = [vp, i]
        L.q3_model_profile_reset.argtypes = [vp]
        L.q3_model_profile_read.argtypes = [vp, i, C.POINTER(C.c_double), C.POINTER(C.c_int64)]
        L.q3_op_matvec.argtypes = [vp, vp, vp, i, i, vp, vp]
        L.q3_session_eval_n.argtypes = [vp, vp, i, i, vp, vp]
        L.q3_op_prefill_attention.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp, i, vp]
        L.q3_model_set_fused_decode.argtypes = [vp, i]
        L.q3_model_fused_decode.argtypes = [vp]
        L.q3_model_set_prefill_tc.argtypes = [vp, i]
        L.q3_model_kv_bytes_per_position.argtypes = [vp]
        L.q3_op_kv_pack_q8_0.argtypes = [vp, i, vp, vp]
        L.q3_op_matvec_affine4.argtypes = [vp, vp, i, i, vp, vp]
        L.q3_model_prefill_tc.argtypes = [vp]
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise Q3Error(rc, lib().q3_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream_handle(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def quantize_q8_0(w: torch.Tensor, stream=None) -> torch.Tensor:
    """Pack a bf16 CUDA tensor [..., n] into canonical Q8_0 blocks (uint8 [..., n/32*34])."""
    assert w.is_cuda and w.dtype == torch.bfloat16 and w.is_contiguous()
    assert w.shape[-1] % 32 == 0
    out = torch.empty(w.shape[:-1] + (w.shape[-1] // 32 * Q8_0_BYTES,), dtype=torch.uint8,
                      device=w.device)
    _check(lib().q3_quantize_q8_0(_ptr(w), w.numel(), _ptr(out), _stream_handle(stream)))
    return out


def quantize_affine4(w: torch.Tensor, stream=None) -> torch.Tensor:
    """Pack a bf16 CUDA tensor [..., n] into AFFINE4_GS32 groups (uint8 [..., n/32*20])."""
    assert w.is_cuda and w.dtype == torch.bfloat16 and w.is_contiguous()
    assert w.shape[-1] % 32 == 0
    out = torch.empty(w.shape[:-1] + (w.shape[-1] // 32 * AFFINE4_BYTES,), dtype=torch.uint8,
                      device=w.device)
    _check(lib().q3_quantize_affine4(_ptr(w), w.numel(), _ptr(out), _stream_handle(stream)))
    return out


def affine4_to_f16(groups: torch.Tensor, n: int, stream=None) -> torch.Tensor:
    """The fp16 copy [..., n] the model keeps of AFFINE4_GS32 groups [..., n/32*20]."""
    assert groups.is_cuda and groups.dtype == torch.uint8 and groups.is_contiguous()
    assert n % 32 == 0 and groups.shape[-1] == n // 32 * AFFINE4_BYTES
    out = torch.empty(groups.shape[:-1] + (n,), dtype=torch.float16, device=groups.device)
    _check(lib().q3_affine4_to_f16(_ptr(groups), out.numel(), _ptr(out), _stream_handle(stream)))
    return out


def op_matmul(w: torch.Tensor, x: torch.Tensor, n: int, block_n: int = 0,
              stream=None) -> torch.Tensor:
    """y[n][m] = sum_k w[m][k] x[n][k] on the tcgen05 GEMM (operator gate).
    w: fp16 [M, K]; x: fp16 [>= round_up(n, 256), K]; block_n: token-tile
    width, 0 for the planner's choice."""
    M, K = w.shape
    assert w.dtype == x.dtype == torch.float16
    assert x.shape[0] >= (n + 255) // 256 * 256 and x.shape[1] == K
    y = torch.empty(n, M, dtype=torch.float32, device=w.device)
    _check(lib().q3_op_matmul(_ptr(w), _ptr(x), M, n, K, _ptr(y), block_n, _stream_handle(stream)))
    return y


NOALLOC_SCRATCH_FLOATS = 2 * 1024 * 1024


OP_STORE, OP_ADD, OP_SWIGLU = 0, 1, 2


def gemm_plan(M: int, N: int, K: int) -> tuple[int, int]:
    """(block_n, k_splits) that a model's rounds use for a projection GEMM of
    M output rows, N token rows and K inputs.  Host only (no GPU)."""
    bn, ks = C.c_int(), C.c_int()
    _check(lib().q3_gemm_plan(M, N, K, C.byref(bn), C.byref(ks)))
    return bn.value, ks.value


def attention_plan(n_kv_heads: int, T: int, max_ctx: int) -> int:
    """Splits per (row, KV head) of the decode attention for T rows whose
    longest context is max_ctx.  Host only (no GPU)."""
    ns = C.c_int()
    _check(lib().q3_attention_plan(n_kv_heads, T, max_ctx, C.byref(ns)))
    return ns.value


def op_gemm(w: torch.Tensor, x: torch.Tensor, n: int, epi: int, out: torch.Tensor,
            w2: torch.Tensor | None = None, block_n: int = 0, k_splits: int = 0,
            stream=None) -> None:
    """One prefill-round projection GEMM with its epilogue and split-K
    (operator gate): OP_STORE out f32 [n, M] = W x; OP_ADD out f32 += W x;
    OP_SWIGLU out fp16 [n, M] = silu(W x) * (W2 x).  w, w2: fp16 [M, K]; x:
    fp16 [>= round_up(n, 256), K].  block_n / k_splits 0: the planner's.
    Synchronous."""
    M, K = w.shape
    if w.dtype != torch.float16 or x.dtype != torch.float16:
        raise ValueError("op_gemm: w and x must be fp16")
    if x.dim() != 2 or x.shape[1] != K or x.shape[0] < (n + 255) // 256 * 256:
        raise ValueError("op_gemm: x must be [>= round_up(n, 256), K]")
    if (epi == OP_SWIGLU) != (w2 is not None) or (w2 is not None and w2.shape != w.shape):
        raise ValueError("op_gemm: OP_SWIGLU takes w2 of w's shape, other epilogues none")
    want = torch.float16 if epi == OP_SWIGLU else torch.float32
    if out.dtype != want or tuple(out.shape) != (n, M):
        raise ValueError(f"op_gemm: out must be {want} [{n}, {M}]")
    ts = [w, x, out] + ([w2] if w2 is not None else [])
    if not all(t.is_contiguous() for t in ts) or len({t.device for t in ts}) != 1:
        raise ValueError("op_gemm: tensors must be contiguous and on one device")
    _check(lib().q3_op_gemm(_ptr(w), _ptr(w2), _ptr(x), M, n, K, epi, _ptr(out), block_n, k_splits,
                            _stream_handle(stream)))


def op_matmul_splitk_noalloc(w: torch.Tensor, x: torch.Tensor, n: int, k_splits: int,
                             y: torch.Tensor, stream=None) -> None:
    """Split-K matmul into the caller's y [n, M] f32 that allocates no device
    memory: the partial sums use the library's fixed scratch array.  For
    callers that cannot allocate at the call site (a framework-owned memory
    pool, a plug-in, a latency-critical loop).  Calls that overlap on the GPU
    race on the shared scratch.  The library cannot see a buffer's extent, so
    the shapes are checked here, before anything is launched: w fp16 [M, K],
    x fp16 [>= round_up(n, 256), K], y f32 [n, M], all contiguous on one
    device.  Returns once the kernels have finished."""
    if w.dim() != 2 or x.dim() != 2 or y.dim() != 2:
        raise ValueError("op_matmul_splitk_noalloc: w, x and y must be 2-D")
    M, K = w.shape
    if w.dtype != torch.float16 or x.dtype != torch.float16 or y.dtype != torch.float32:
        raise ValueError("op_matmul_splitk_noalloc: w and x fp16, y float32")
    if x.shape[1] != K or x.shape[0] < (n + 255) // 256 * 256:
        raise ValueError(f"op_matmul_splitk_noalloc: x must be [>= {(n + 255) // 256 * 256}, {K}]")
    if tuple(y.shape) != (n, M):
        raise ValueError(f"op_matmul_splitk_noalloc: y must be [{n}, {M}]")
    if not (w.is_contiguous() and x.is_contiguous() and y.is_contiguous()):
        raise ValueError("op_matmul_splitk_noalloc: tensors must be contiguous")
    if not (w.device == x.device == y.device) or w.device.type != "cuda":
        raise ValueError("op_matmul_splitk_noalloc: tensors must be on one CUDA device")
    rc = lib().q3_op_matmul_splitk_noalloc(_ptr(w), _ptr(x), M, n, K, k_splits, _ptr(y),
                                           _stream_handle(stream))
    if rc != 0:
        raise Q3Error(rc, lib().q3_noalloc_last_error().decode())


def op_kv_pack_q8_0(rows: torch.Tensor, stream=None) -> torch.Tensor:
    """The Q8_0 cache writers' packing of f32 rows [n, 128] into canonical
    Q8_0 blocks (uint8 [n, 136]) (operator gate)."""
    if rows.dtype != torch.float32 or rows.dim() != 2 or rows.shape[1] != 128 or not rows.is_contiguous():
        raise ValueError("op_kv_pack_q8_0: rows must be contiguous float32 [n, 128]")
    out = torch.empty(rows.shape[0], 136, dtype=torch.uint8, device=rows.device)
    _check(lib().q3_op_kv_pack_q8_0(_ptr(rows), rows.shape[0], _ptr(out), _stream_handle(stream)))
    return out


def op_matvec(w: torch.Tensor, x: torch.Tensor, scales: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """y[m] = sum_k w[m][k] x[k] on the decode GEMV (operator gate).  w: bf16
    [M, K], or the int8 quant plane with scales the fp16 [M, K/32] plane."""
    M, K = w.shape
    y = torch.empty(M, dtype=torch.float32, device=w.device)
    _check(lib().q3_op_matvec(_ptr(w), _ptr(scales), _ptr(x), M, K, _ptr(y),
                              _stream_handle(stream)))
    return y


def op_matvec_affine4(groups: torch.Tensor, x: torch.Tensor, M: int, K: int, stream=None) -> torch.Tensor:
    """y[m] = sum_k w[m][k] x[k] on the 5.0-bit AFFINE4 matvec (operator gate):
    groups uint8 [M, K/32*20] (q3_quantize_affine4's format), x f32 [K].
    Synchronous."""
    if groups.dtype != torch.uint8 or groups.numel() != M * K // 32 * AFFINE4_BYTES or not groups.is_contiguous():
        raise ValueError("op_matvec_affine4: groups must be contiguous uint8 [M, K/32*20]")
    if x.dtype != torch.float32 or x.numel() != K or not x.is_contiguous():
        raise ValueError("op_matvec_affine4: x must be contiguous float32 [K]")
    y = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(lib().q3_op_matvec_affine4(_ptr(groups), _ptr(x), M, K, _ptr(y), _stream_handle(stream)))
    return y


def op_prefill_attention(q: torch.Tensor, kv: torch.Tensor, table: torch.Tensor, pos0: int,
                         n_kv: int, use_tc: bool = True, stream=None) -> torch.Tensor:
    """Causal GQA attention of one session's prefill round over its paged K/V
    (operator gate of the prefill attention).  q: fp16 [T, n_q, 128]; kv:
    bf16 [n_blocks, 2, n_kv, 32, 128]; table: int32 physical block of each 32
    positions.  Returns fp16 [T, n_q * 128].  Synchronous."""
    T, n_q, d = q.shape
    assert d == 128 and q.dtype == torch.float16 and kv.dtype == torch.bfloat16
    assert table.dtype == torch.int32
    out = torch.empty(T, n_q * 128, dtype=torch.float16, device=q.device)
    _check(lib().q3_op_prefill_attention(_ptr(q), _ptr(kv), _ptr(table), table.numel(), kv.shape[0],
                                         pos0, T, n_q, n_kv, _ptr(out), 1 if use_tc else 0,
                                         _stream_handle(stream)))
    return out


class Model:
    """A decoder over device weights (synthetic.make_weights() layout).

    weights: {"embed", "final_norm", "lm_head" (None if tied), "layers": [...]};
    for a Q8_0 shape the seven projections of each layer must be canonical
    Q8_0 blocks (uint8), e.g. from quantize_q8_0, and for an AFFINE4 shape
    AFFINE4_GS32 groups (uint8), e.g. from quantize_affine4.  The tensors are
    borrowed and kept referenced by this object.
    """

    def __init__(self, shape, weights: dict, max_ctx: int, max_round_tokens: int = 2048,
                 stream=None):
        kv_scheme = getattr(shape, "kv_quant", BF16)
        if kv_scheme not in (BF16, Q8_0):
            raise ValueError(f"unknown K/V cache scheme {kv_scheme}")
        self.shape = shape
        self.stream = stream or torch.cuda.current_stream()
        self._keep = weights
        cfg = _Config(shape.n_layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads,
                      shape.head_dim, shape.ffn, shape.vocab, max_ctx, shape.rope_theta,
                      shape.rms_eps, int(shape.tied), shape.scheme, kv_scheme)
        layers = (_LayerW * shape.n_layers)()
        for li, lw in enumerate(weights["layers"]):
            for name in ("attn_norm", "q_norm", "k_norm", "ffn_norm") + PROJ:
                t = lw[name]
                assert t.is_cuda and t.is_contiguous(), name
                setattr(layers[li], name, t.data_ptr())
        self._layers = layers
        lm = weights.get("lm_head")
        w = _Weights(weights["embed"].data_ptr(), weights["final_norm"].data_ptr(),
                     lm.data_ptr() if lm is not None else None, layers)
        h = C.c_void_p()
        _check(lib().q3_model_create(C.byref(cfg), C.byref(w), max_round_tokens,
                                     _stream_handle(self.stream), C.byref(h)))
        self.h = h
        self.max_ctx = max_ctx
        self.max_round_tokens = max_round_tokens

    def close(self):
        if getattr(self, "h", None):
            lib().q3_model_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def pool(self, n_blocks: int, max_sessions: int = 64) -> "Pool":
        return Pool(self, n_blocks, max_sessions)

    def sync(self) -> None:
        _check(lib().q3_sync(self.h))

    @property
    def kv_bytes_per_position(self) -> int:
        """Bytes one position's K and V take in one layer of the cache."""
        return lib().q3_model_kv_bytes_per_position(self.h)

    @property
    def launch_count(self) -> int:
        return lib().q3_model_launch_count(self.h)

    KERNEL_CLASSES = ("gemv", "gemm", "attention", "qk_norm_rope_append", "norm", "other",
                      "decode_step")

    @property
    def fused_decode(self) -> bool:
        """Whether one-session decode rounds run as the one-kernel fused step."""
        return bool(lib().q3_model_fused_decode(self.h))

    def set_fused_decode(self, on: bool) -> None:
        """Select the fused decode step (default where supported) or the per-operation path."""
        _check(lib().q3_model_set_fused_decode(self.h, 1 if on else 0))

    @property
    def prefill_tc(self) -> bool:
        """True when prefill attention runs on the tcgen05 kernel."""
        return bool(lib().q3_model_prefill_tc(self.h))

    def set_prefill_tc(self, on: bool) -> None:
        """Choose the tcgen05 (True) or mma.sync (False) prefill attention."""
        _check(lib().q3_model_set_prefill_tc(self.h, 1 if on else 0))

    def profile(self, on: bool) -> None:
        """Per-launch CUDA-event timing by kernel class (serialises launches)."""
        _check(lib().q3_model_profile(self.h, int(on)))

    def profile_reset(self) -> None:
        _check(lib().q3_model_profile_reset(self.h))

    def profile_read(self) -> dict:
        """{class: (total device ms, launches)} since the last reset."""
        out = {}
        for i, name in enumerate(self.KERNEL_CLASSES):
            ms, n = C.c_double(), C.c_int64()
            _check(lib().q3_model_profile_read(self.h, i, C.byref(ms), C.byref(n)))
            out[name] = (ms.value, n.value)
        return out

    def eval_batch(self, sessions, tokens: torch.Tensor, n, logits: torch.Tensor,
                   argmax: torch.Tensor | None = None) -> None:
        """One round over several sessions: tokens (int32, device) concatenated
        in session order; logits [ns, vocab] f32 device; argmax [ns] int32."""
        ns = len(sessions)
        hs = (C.c_void_p * ns)(*[s.h.value for s in sessions])
        nn = (C.c_int * ns)(*[int(k) for k in n])
        _check(lib().q3_eval_batch(hs, ns, _ptr(tokens), nn, _ptr(logits), _ptr(argmax)))


class Pool:
    def __init__(self, model: Model, n_blocks: int, max_sessions: int):
        self.model = model
        h = C.c_void_p()
        _check(lib().q3_pool_create(model.h, n_blocks, max_sessions, C.byref(h)))
        self.h = h
        self.n_blocks = n_blocks

    def close(self):
        if getattr(self, "h", None):
            lib().q3_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def session(self) -> "Session":
        return Session(self)

    def enable_prefix(self, hash_bits: int = 16) -> None:
        """Content-addressed prefix sharing over this pool (2^hash_bits buckets)."""
        _check(lib().q3_pool_enable_prefix(self.h, hash_bits))


class Session:
    def __init__(self, pool: Pool):
        self.pool = pool
        h = C.c_void_p()
        _check(lib().q3_session_create(pool.h, C.byref(h)))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().q3_session_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_block_table(self, ids) -> None:
        import numpy as np
        a = np.ascontiguousarray(ids, np.int32)
        _check(lib().q3_session_set_block_table(self.h, a.ctypes.data_as(C.c_void_p), a.size))

    def publish(self, tokens) -> int:
        """Share the session's full blocks; tokens (host) are those it evaluated.
        Returns how many blocks were newly published."""
        import numpy as np
        a = np.ascontiguousarray(tokens, np.int32)
        out = C.c_int(0)
        _check(lib().q3_session_publish(self.h, a.ctypes.data_as(C.c_void_p), a.size, C.byref(out)))
        return out.value

    def attach_prefix(self, tokens) -> int:
        """On an empty session: attach the longest published chain matching the
        prompt's leading full blocks; returns the positions attached."""
        import numpy as np
        a = np.ascontiguousarray(tokens, np.int32)
        out = C.c_int(0)
        _check(lib().q3_session_attach_prefix(self.h, a.ctypes.data_as(C.c_void_p), a.size, C.byref(out)))
        return out.value

    def eval_n(self, tokens: torch.Tensor, n_logits: int, logits: torch.Tensor,
               argmax: torch.Tensor | None = None) -> None:
        """Append a round of tokens and write the logits of its last n_logits
        rows: logits [n_logits, vocab] f32 device, argmax [n_logits] int32."""
        assert tokens.is_cuda and tokens.dtype == torch.int32 and tokens.is_contiguous()
        assert logits.is_contiguous() and logits.numel() >= n_logits * logits.shape[-1]
        _check(lib().q3_session_eval_n(self.h, _ptr(tokens), tokens.numel(), n_logits, _ptr(logits),
                                       _ptr(argmax)))

    def eval(self, tokens: torch.Tensor, logits: torch.Tensor,
             argmax: torch.Tensor | None = None) -> None:
        """Append a round of tokens (int32, device); logits [vocab] f32 device."""
        assert tokens.is_cuda and tokens.dtype == torch.int32 and tokens.is_contiguous()
        _check(lib().q3_session_eval(self.h, _ptr(tokens), tokens.numel(), _ptr(logits),
                                     _ptr(argmax)))

    def truncate(self, n_pos: int) -> None:
        _check(lib().q3_session_truncate(self.h, n_pos))

    def reset(self) -> None:
        _check(lib().q3_session_reset(self.h))

    @property
    def pos(self) -> int:
        return lib().q3_session_pos(self.h)


def device_weights(shape, weights: dict) -> dict:
    """The weight dict the library takes: bf16 tensors as given; for a Q8_0
    or AFFINE4 shape the seven projections packed by the library's own
    quantizer (q3_quantize_q8_0, q3_quantize_affine4)."""
    if shape.scheme not in (Q8_0, AFFINE4):
        return weights
    pack = quantize_q8_0 if shape.scheme == Q8_0 else quantize_affine4
    out = dict(weights)
    out["layers"] = []
    for lw in weights["layers"]:
        d = dict(lw)
        for name in PROJ:
            d[name] = pack(lw[name])
        out["layers"].append(d)
    return out
