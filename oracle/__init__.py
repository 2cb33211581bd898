"""Plain CPU oracle for the dense Qwen3-style decoder forward (ctypes binding).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg import this package.  It shares no code with the
CUDA path (qwen3_dense_decoder_gb300) and never imports it.

The C source (q3_oracle.c) states what each function follows on the Kipp
pages.  ``build()`` compiles it with gcc into this directory.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q3_oracle.c")
_HDR = os.path.join(_HERE, "q3_oracle.h")
_LIB = os.path.join(_HERE, "libq3_oracle.so")

BF16, Q8_0, AFFINE4 = 0, 1, 2
BLOCK = 32
Q8_0_BYTES = 34
AFFINE4_BYTES = 20


def build(force: bool = False) -> str:
    """Compile the oracle shared library if missing or stale; return its path."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared",
                               "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("hidden", C.c_int), ("n_q_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("tied", C.c_int), ("scheme", C.c_int),
                ("rope_theta", C.c_double), ("rms_eps", C.c_double), ("kv_quant", C.c_int)]


class _Layer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("attn_norm", "q_norm", "k_norm", "ffn_norm",
                 "wq", "wk", "wv", "wo", "wg", "wu", "wd")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        vp, i, d, f = C.c_void_p, C.c_int, C.c_double, C.c_float
        L.orc_bf16_to_f32.argtypes, L.orc_bf16_to_f32.restype = [C.c_uint16], f
        L.orc_f32_to_bf16.argtypes, L.orc_f32_to_bf16.restype = [f], C.c_uint16
        L.orc_f16_to_f32.argtypes, L.orc_f16_to_f32.restype = [C.c_uint16], f
        L.orc_f32_to_f16.argtypes, L.orc_f32_to_f16.restype = [f], C.c_uint16
        L.orc_q8_0_pack.argtypes = [vp, C.c_long, vp]
        L.orc_q8_0_unpack.argtypes = [vp, C.c_long, vp]
        L.orc_affine4_pack.argtypes = [vp, C.c_long, vp]
        L.orc_affine4_unpack.argtypes = [vp, C.c_long, vp]
        L.orc_rmsnorm.argtypes = [vp, vp, i, d, vp]
        L.orc_rope.argtypes = [vp, i, i, d]
        L.orc_silu.argtypes, L.orc_silu.restype = [f], f
        L.orc_matmul.argtypes = [vp, i, i, i, vp, i, vp, i]
        L.orc_gqa_attend.argtypes = [vp, vp, vp, i, i, i, i, vp]
        L.orc_model_create.argtypes = [C.POINTER(_Cfg), vp, vp, vp, C.POINTER(_Layer), i]
        L.orc_model_create.restype = vp
        L.orc_model_free.argtypes = [vp]
        L.orc_pool_create.argtypes, L.orc_pool_create.restype = [vp, i], vp
        L.orc_pool_free.argtypes = [vp]
        L.orc_session_create.argtypes, L.orc_session_create.restype = [vp, vp, i], vp
        L.orc_session_free.argtypes = [vp]
        L.orc_session_set_block_table.argtypes = [vp, vp, i]
        L.orc_session_pos.argtypes = [vp]
        L.orc_session_truncate.argtypes = [vp, i]
        L.orc_eval.argtypes = [vp, vp, i, vp, vp]
        L.orc_eval_batch.argtypes = [vp, vp, vp, i, vp]
        L.orc_eval_rows.argtypes = [vp, vp, i, vp, i, vp]
        L.orc_argmax.argtypes = [vp, i]
        L.orc_pool_enable_prefix.argtypes = [vp, i]
        L.orc_session_publish.argtypes = [vp]
        L.orc_pool_free_blocks.argtypes = [vp]
        L.orc_session_attach_prefix.argtypes = [vp, vp, i]
        L.orc_kv_bytes_per_position.argtypes = [C.POINTER(_Cfg)]
        L.orc_kv_bytes_per_position.restype = C.c_long
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


# ---------------------------------------------------------------- components

def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a torch bf16 tensor (no arithmetic)."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32).ravel()
    return np.array([lib().orc_f32_to_bf16(float(v)) for v in x], np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, np.uint16).ravel()
    return np.array([lib().orc_bf16_to_f32(int(v)) for v in b], np.float32)


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32).ravel()
    return np.array([lib().orc_f32_to_f16(float(v)) for v in x], np.uint16)


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, np.uint16).ravel()
    return np.array([lib().orc_f16_to_f32(int(v)) for v in h], np.float32)


def q8_0_pack(w: np.ndarray) -> np.ndarray:
    """float32 weights [..., n] (n % 32 == 0) -> canonical 34-byte blocks (uint8)."""
    w = np.ascontiguousarray(w, np.float32)
    assert w.shape[-1] % BLOCK == 0
    out = np.empty(w.shape[:-1] + (w.shape[-1] // BLOCK * Q8_0_BYTES,), np.uint8)
    lib().orc_q8_0_pack(_ptr(w), w.size, _ptr(out))
    return out


def q8_0_unpack(blocks: np.ndarray, n: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, np.uint8)
    out = np.empty(blocks.shape[:-1] + (n,), np.float32)
    lib().orc_q8_0_unpack(_ptr(blocks), out.size, _ptr(out))
    return out


def affine4_pack(w: np.ndarray) -> np.ndarray:
    """float32 weights [..., n] (n % 32 == 0) -> 20-byte AFFINE4_GS32 groups (uint8)."""
    w = np.ascontiguousarray(w, np.float32)
    assert w.shape[-1] % BLOCK == 0
    out = np.empty(w.shape[:-1] + (w.shape[-1] // BLOCK * AFFINE4_BYTES,), np.uint8)
    lib().orc_affine4_pack(_ptr(w), w.size, _ptr(out))
    return out


def affine4_unpack(groups: np.ndarray, n: int) -> np.ndarray:
    groups = np.ascontiguousarray(groups, np.uint8)
    out = np.empty(groups.shape[:-1] + (n,), np.float32)
    lib().orc_affine4_unpack(_ptr(groups), out.size, _ptr(out))
    return out


def rmsnorm(x: np.ndarray, gain_bits: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    g = np.ascontiguousarray(gain_bits, np.uint16)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_ptr(x), _ptr(g), x.size, eps, _ptr(y))
    return y


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, np.float32, copy=True)
    lib().orc_rope(_ptr(v), v.size, pos, theta)
    return v


def silu(z: float) -> float:
    return lib().orc_silu(z)


def matmul(W: np.ndarray, scheme: int, n_out: int, n_in: int, x: np.ndarray,
           n_threads: int = 1) -> np.ndarray:
    W = np.ascontiguousarray(W)
    x = np.ascontiguousarray(x, np.float32).reshape(-1, n_in)
    y = np.empty((x.shape[0], n_out), np.float32)
    lib().orc_matmul(_ptr(W), scheme, n_out, n_in, _ptr(x), x.shape[0], _ptr(y), n_threads)
    return y


def gqa_attend(q: np.ndarray, K_bits: np.ndarray, V_bits: np.ndarray, n_q: int,
               n_kv: int, d: int) -> np.ndarray:
    """q [n_q, d] f32; K, V [ctx, n_kv, d] bf16 bits -> o [n_q, d]."""
    q = np.ascontiguousarray(q, np.float32)
    K = np.ascontiguousarray(K_bits, np.uint16)
    V = np.ascontiguousarray(V_bits, np.uint16)
    o = np.empty((n_q, d), np.float32)
    lib().orc_gqa_attend(_ptr(q), _ptr(K), _ptr(V), K.shape[0], n_q, n_kv, d, _ptr(o))
    return o


def argmax(v: np.ndarray) -> int:
    v = np.ascontiguousarray(v, np.float32)
    return lib().orc_argmax(_ptr(v), v.size)


# ---------------------------------------------------------------- model

def _cfg(shape) -> _Cfg:
    return _Cfg(shape.n_layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads,
                shape.head_dim, shape.ffn, shape.vocab, int(shape.tied), shape.scheme,
                shape.rope_theta, shape.rms_eps, getattr(shape, "kv_quant", BF16))


def kv_bytes_per_position(shape) -> int:
    """Bytes one position's K and V take in one layer's cache (bf16 or Q8_0)."""
    cfg = _cfg(shape)
    return lib().orc_kv_bytes_per_position(C.byref(cfg))


class Model:
    """Oracle model over host copies of the synthetic weights.

    ``weights`` is synthetic.make_weights()'s dict (torch bf16 tensors, any
    device).  For a Q8_0 or AFFINE4 shape the oracle packs the seven
    projections itself with its own packer (``packed`` keeps them per layer).
    """

    PROJ = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")

    def __init__(self, shape, weights: dict, n_threads: int | None = None):
        self.shape = shape
        self.n_threads = n_threads or default_threads()
        self._keep = []

        def keep(a):
            self._keep.append(a)
            return a.ctypes.data

        self.embed = bf16_bits(weights["embed"])
        emb = keep(self.embed)
        fnorm = keep(bf16_bits(weights["final_norm"]))
        lm = keep(bf16_bits(weights["lm_head"])) if not shape.tied else None
        self.packed = []      # per layer {name: blocks or groups} when quantized
        layers = (_Layer * shape.n_layers)()
        for li, lw in enumerate(weights["layers"]):
            ptrs = {}
            for name in ("attn_norm", "q_norm", "k_norm", "ffn_norm"):
                ptrs[name] = keep(bf16_bits(lw[name]))
            packed = {}
            for name in self.PROJ:
                bits = bf16_bits(lw[name])
                if shape.scheme in (Q8_0, AFFINE4):
                    pack = q8_0_pack if shape.scheme == Q8_0 else affine4_pack
                    blk = pack(bf16_to_f32_fast(bits).reshape(bits.shape))
                    packed[name] = blk
                    ptrs[name] = keep(blk)
                else:
                    ptrs[name] = keep(bits)
            self.packed.append(packed)
            L = layers[li]
            L.attn_norm, L.q_norm, L.k_norm, L.ffn_norm = (
                ptrs["attn_norm"], ptrs["q_norm"], ptrs["k_norm"], ptrs["ffn_norm"])
            L.wq, L.wk, L.wv, L.wo = ptrs["wq"], ptrs["wk"], ptrs["wv"], ptrs["wo"]
            L.wg, L.wu, L.wd = ptrs["w_gate"], ptrs["w_up"], ptrs["w_down"]
        cfg = _cfg(shape)
        self._layers = layers
        self.h = lib().orc_model_create(C.byref(cfg), emb, fnorm, lm, layers, self.n_threads)
        if not self.h:
            raise ValueError("oracle: bad shape")

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_model_free(self.h)
            self.h = None

    def pool(self, n_blocks: int) -> "Pool":
        return Pool(self, n_blocks)

    def session(self, pool: "Pool | None" = None, max_ctx: int = 4096) -> "Session":
        return Session(self, pool, max_ctx)

    def eval_batch(self, sessions, token_lists) -> np.ndarray:
        ns = len(sessions)
        arrs = [np.ascontiguousarray(t, np.int32) for t in token_lists]
        hs = (C.c_void_p * ns)(*[s.h for s in sessions])
        tp = (C.c_void_p * ns)(*[a.ctypes.data for a in arrs])
        n = (C.c_int * ns)(*[a.size for a in arrs])
        out = np.empty((ns, self.shape.vocab), np.float32)
        if lib().orc_eval_batch(hs, tp, n, ns, _ptr(out)):
            raise RuntimeError("oracle: eval_batch failed")
        return out


def bf16_to_f32_fast(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 by placing them in the upper half (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


class Pool:
    def __init__(self, model: Model, n_blocks: int):
        self.model = model
        self.h = lib().orc_pool_create(model.h, n_blocks)
        if not self.h:
            raise MemoryError("oracle: pool")

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_pool_free(self.h)
            self.h = None

    @property
    def free_blocks(self) -> int:
        return lib().orc_pool_free_blocks(self.h)

    def enable_prefix(self, hash_bits: int = 16) -> None:
        """Content-addressed prefix sharing over this pool (2^hash_bits buckets)."""
        if lib().orc_pool_enable_prefix(self.h, hash_bits):
            raise ValueError("oracle: enable_prefix")


class Session:
    def __init__(self, model: Model, pool: Pool | None, max_ctx: int):
        self.model, self.pool = model, pool
        self.h = lib().orc_session_create(model.h, pool.h if pool else None, max_ctx)
        if not self.h:
            raise MemoryError("oracle: session")

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_session_free(self.h)
            self.h = None

    def set_block_table(self, ids) -> None:
        ids = np.ascontiguousarray(ids, np.int32)
        if lib().orc_session_set_block_table(self.h, _ptr(ids), ids.size):
            raise ValueError("oracle: bad block table")

    def publish(self) -> int:
        """Make the session's full blocks shareable; returns how many were newly published."""
        n = lib().orc_session_publish(self.h)
        if n < 0:
            raise ValueError("oracle: publish")
        return n

    def attach_prefix(self, tokens) -> int:
        """At position 0: attach the longest published chain matching the prompt's
        leading full blocks (at least one token left); returns the positions attached."""
        t = np.ascontiguousarray(tokens, np.int32)
        n = lib().orc_session_attach_prefix(self.h, _ptr(t), t.size)
        if n < 0:
            raise ValueError("oracle: attach_prefix")
        return n

    @property
    def pos(self) -> int:
        return lib().orc_session_pos(self.h)

    def truncate(self, n_pos: int) -> None:
        if lib().orc_session_truncate(self.h, n_pos):
            raise ValueError("oracle: bad truncate")

    def eval(self, tokens, all_rows: bool = False) -> np.ndarray:
        """Logits of the round's last row [vocab], or of every row [n, vocab]."""
        t = np.ascontiguousarray(tokens, np.int32)
        V = self.model.shape.vocab
        last = np.empty(V, np.float32)
        allr = np.empty((t.size, V), np.float32) if all_rows else None
        rc = lib().orc_eval(self.h, _ptr(t), t.size, _ptr(last),
                            _ptr(allr) if all_rows else None)
        if rc:
            raise RuntimeError("oracle: eval failed (capacity or token range)")
        return allr if all_rows else last

    def eval_rows(self, tokens, rows) -> np.ndarray:
        """Logits [len(rows), vocab] of the listed rows of the round (indices
        into tokens, increasing); an empty list appends the positions and
        computes no logits."""
        t = np.ascontiguousarray(tokens, np.int32)
        r = np.ascontiguousarray(rows, np.int32)
        out = np.empty((r.size, self.model.shape.vocab), np.float32)
        rc = lib().orc_eval_rows(self.h, _ptr(t), t.size, _ptr(r) if r.size else None, r.size,
                                 _ptr(out) if r.size else None)
        if rc:
            raise RuntimeError("oracle: eval_rows failed (capacity, token range or row list)")
        return out

    def append(self, tokens) -> None:
        """Append a round's positions (K/V stored) without computing logits."""
        self.eval_rows(tokens, [])


def nmse(got: np.ndarray, ref: np.ndarray) -> float:
    """sum (g - o)^2 / sum o^2 with o the oracle's logits."""
    g = np.asarray(got, np.float64)
    o = np.asarray(ref, np.float64)
    return float(((g - o) ** 2).sum() / (o ** 2).sum())
