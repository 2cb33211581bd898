"""Seeded synthetic inputs shared by the CUDA path's tests and bench and by the oracle.

This module holds no arithmetic of the decoder: it only draws random numbers
(weights, prompt tokens, block-table permutations, prompt lengths) and states
the model shapes.  Both sides receive the same bytes from here.

Shapes follow the dense Qwen3 family as the Kipp pages describe it ("Kipp Model
Support", section "The registry": 8 KV heads, head width 128, vocabulary
151,936, RMS epsilon 1e-6, per-checkpoint RoPE theta and embedding tying).
Recipe: projections, embedding and an untied lm_head are bf16(N(0, 0.02));
norm gains are bf16(1 + N(0, 0.02)); each tensor draws from its own generator
seeded with base_seed + its index in a fixed order.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

BF16, Q8_0, AFFINE4 = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    tied: bool
    scheme: int = BF16
    rope_theta: float = 1e6
    rms_eps: float = 1e-6
    kv_quant: int = BF16      # K/V cache: BF16, or Q8_0 blocks (the opt-in quantized cache)

    @property
    def q_width(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim

    def replace(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


SHAPES = {
    # 2 layers, hidden 1024, 16/8 heads of 128, FFN 3072, vocab 4096, tied
    "tiny": Shape("tiny", 2, 1024, 16, 8, 128, 3072, 4096, True),
    "0.6b": Shape("qwen3-0.6b", 28, 1024, 16, 8, 128, 3072, 151936, True),
    "4b": Shape("qwen3-4b", 36, 2560, 32, 8, 128, 9728, 151936, True),
    "8b-q8_0": Shape("qwen3-8b-q8_0", 36, 4096, 32, 8, 128, 12288, 151936, False, Q8_0),
    "4b-affine4": Shape("qwen3-4b-affine4", 36, 2560, 32, 8, 128, 9728, 151936, True, AFFINE4),
    "14b": Shape("qwen3-14b", 40, 5120, 40, 8, 128, 17408, 151936, False),
}

LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
                 "ffn_norm", "w_gate", "w_up", "w_down")
NORM_TENSORS = ("attn_norm", "q_norm", "k_norm", "ffn_norm")


def layer_tensor_shape(s: Shape, name: str) -> tuple[int, ...]:
    return {
        "attn_norm": (s.hidden,), "ffn_norm": (s.hidden,),
        "q_norm": (s.head_dim,), "k_norm": (s.head_dim,),
        "wq": (s.q_width, s.hidden), "wk": (s.kv_width, s.hidden),
        "wv": (s.kv_width, s.hidden), "wo": (s.hidden, s.q_width),
        "w_gate": (s.ffn, s.hidden), "w_up": (s.ffn, s.hidden),
        "w_down": (s.hidden, s.ffn),
    }[name]


def _draw(shape, seed: int, device, gain: bool) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 0.02
    if gain:
        w += 1.0
    return w.to(torch.bfloat16)


def make_weights(s: Shape, seed: int = 1234, device="cpu") -> dict:
    """bf16 weights for shape s: {"embed", "final_norm", "lm_head" (None if tied),
    "layers": [{name: tensor}]}.  For a Q8_0 or AFFINE4 shape these are the
    bf16 source weights that the quantizers of either side pack."""
    k = seed
    out = {"embed": _draw((s.vocab, s.hidden), k, device, False)}
    k += 1
    out["final_norm"] = _draw((s.hidden,), k, device, True)
    k += 1
    out["lm_head"] = None
    if not s.tied:
        out["lm_head"] = _draw((s.vocab, s.hidden), k, device, False)
    k += 1
    layers = []
    for _ in range(s.n_layers):
        lw = {}
        for name in LAYER_TENSORS:
            lw[name] = _draw(layer_tensor_shape(s, name), k, device, name in NORM_TENSORS)
            k += 1
        layers.append(lw)
    out["layers"] = layers
    return out


def make_tokens(n: int, vocab: int, seed: int) -> np.ndarray:
    """n prompt tokens drawn uniformly from [0, vocab)."""
    return np.random.default_rng(seed).integers(0, vocab, size=n, dtype=np.int32)


def make_block_permutation(n_blocks: int, seed: int) -> np.ndarray:
    """A seeded random permutation of the pool's block ids."""
    return np.random.default_rng(seed).permutation(n_blocks).astype(np.int32)


def make_prompt_lengths(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n prompt lengths uniform in [lo, hi]."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=n).astype(np.int32)
