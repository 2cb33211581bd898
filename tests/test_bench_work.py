"""The algorithmic work the benchmark divides by, pinned to the shapes'
registry figures ("Kipp Model Support", section "The registry": layers,
hidden, heads, FFN, vocabulary, tying) worked out by hand from the dense
Qwen3 layer (Q/K/V/O and gate/up/down projections, head width 128).

- projection parameters per shape, and the decode-step bytes: every
  projection once (2 B per BF16 weight, 34 B per 32 Q8_0 weights), the
  lm_head once (BF16), and 2 x n_kv x 128 x 2 B of K/V per layer per cached
  position;
- prefill FLOPs: 2 x params x tokens, causal QK^T and PV over T^2/2 pairs
  (4 x 128 x n_q x L x T^2 / 2), and one lm_head row.
"""
import bench
import synthetic

S = synthetic.SHAPES


def test_projection_parameters():
    # 4B: per layer (4096 + 2 x 1024) x 2560 + 2560 x 4096 + 3 x 9728 x 2560
    assert bench.proj_params(S["4b"]) == 36 * (6144 * 2560 + 2560 * 4096 + 3 * 9728 * 2560) == 3_633_315_840
    assert bench.proj_params(S["0.6b"]) == 28 * (4096 * 1024 + 1024 * 2048 + 3 * 3072 * 1024) == 440_401_920
    assert bench.proj_params(S["8b-q8_0"]) == 36 * (6144 * 4096 + 4096 * 4096 + 3 * 12288 * 4096) == 6_945_767_424
    assert bench.proj_params(S["14b"]) == 40 * (7168 * 5120 + 5120 * 5120 + 3 * 17408 * 5120) == 13_212_057_600


def test_decode_step_bytes():
    s4 = S["4b"]
    w4 = 2 * 3_633_315_840 + 2 * 151_936 * 2560                # 8.045 GB
    assert abs(bench.step_bytes(s4, [0]) - w4) < 1
    assert abs(bench.decode_bytes(s4, 0) - w4) < 1
    # K/V per cached position: 36 layers x 2 x 1024 x 2 B = 147,456 B
    assert abs(bench.step_bytes(s4, [1000]) - w4 - 147_456 * 1000) < 1
    assert abs(bench.decode_bytes(s4, 10, batch=3) - w4 - 147_456 * 30) < 1
    # Q8_0 projections at 34 B per 32 weights, untied BF16 lm_head: 8.62 GB
    s8 = S["8b-q8_0"]
    w8 = 6_945_767_424 * 34 / 32 + 2 * 151_936 * 4096
    assert abs(bench.step_bytes(s8, [0]) - w8) < 1 and 8.61e9 < w8 < 8.63e9
    # AFFINE4_GS32 projections at 20 B per 32 weights, tied BF16 lm_head: 3.05 GB
    sa = S["4b-affine4"]
    wa = 3_633_315_840 * 20 / 32 + 2 * 151_936 * 2560
    assert abs(bench.step_bytes(sa, [0]) - wa) < 1 and 3.04e9 < wa < 3.05e9
    # 14B: 27.98 GB of weights, 163,840 B of K/V per position (40 layers)
    s14 = S["14b"]
    w14 = 2 * 13_212_057_600 + 2 * 151_936 * 5120
    assert abs(bench.step_bytes(s14, [7, 9]) - w14 - 163_840 * 16) < 1 and 27.9e9 < w14 < 28.0e9


def test_prefill_flops():
    s4 = S["4b"]
    T = 2048
    attn = 4 * 128 * 32 * 36 * T * T / 2
    ref = 2 * 3_633_315_840 * T + attn + 2 * 151_936 * 2560
    assert abs(bench.prefill_flops(s4, T) - ref) < 1e3
    assert 16.11e12 < ref < 16.13e12                            # 16.12 TFLOP
