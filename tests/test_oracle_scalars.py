"""Pins of the oracle's scalar conversions and of its Q8_0 and AFFINE4_GS32 packers.

bf16 and fp16 rounding are checked against library conversions that
implement the same IEEE rules (torch's bf16 cast, numpy's float16 cast);
Q8_0 against blocks worked by hand (tests/golden/q8_0_worked_example.json)
and against closed-form error bounds of the format ("Kipp Model Support",
section "Quantization (Q8_0)"); AFFINE4_GS32 against groups worked by hand
(tests/golden/affine4_gs32_worked_example.json) and against the closed forms
of rounding to a 16-point grid ("Kipp Model Support", section
"Quantization (AFFINE4_GS32)").
"""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _edge_floats():
    vals = [0.0, -0.0, 1.0, -1.0, 1.5, 3.0e38, -3.0e38, 1e-40, -1e-40, 1e-45,
            65504.0, 65519.99, 65520.0, 65536.0, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8,
            float("inf"), float("-inf")]
    # exact bf16 ties: 1 + 2^-8 (tie, even below), 1 + 3 * 2^-8 (tie, even above)
    vals += [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)]
    # exact fp16 ties: 1 + 2^-11, 1 + 3 * 2^-11, subnormal tie 2^-25
    vals += [1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2.0 ** -25, 3 * 2.0 ** -25]
    return np.array(vals, np.float32)


def test_bf16_round_nearest_even_matches_torch(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([_edge_floats(),
                        rng.standard_normal(4000).astype(np.float32) * 0.02,
                        (rng.standard_normal(2000) * 1e4).astype(np.float32),
                        rng.uniform(-1, 1, 2000).astype(np.float32) * 1e-38])
    ours = orc.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # and back: the bf16 value is the upper half of the float
    back = orc.bf16_to_f32(ref)
    np.testing.assert_array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                                  .float().numpy())


def test_fp16_conversions_match_ieee(orc):
    rng = np.random.default_rng(1)
    x = np.concatenate([_edge_floats(), rng.standard_normal(4000).astype(np.float32) * 0.02 / 127,
                        rng.standard_normal(2000).astype(np.float32) * 100,
                        rng.uniform(0, 1e-4, 2000).astype(np.float32)])
    ours = orc.f32_to_f16(x)
    ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # decode every finite pattern
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite(allbits.view(np.float16))
    dec = orc.f16_to_f32(allbits[finite])
    np.testing.assert_array_equal(dec, allbits[finite].view(np.float16).astype(np.float32))


def test_q8_0_hand_worked_blocks(orc):
    spec = json.load(open(os.path.join(GOLDEN, "q8_0_worked_example.json")))
    for blk in spec["blocks"]:
        w = np.array(blk["k_times_2pow_minus10"], np.float64) * 2.0 ** -10
        w = w.astype(np.float32)
        assert np.all(w.astype(np.float64) == np.array(blk["k_times_2pow_minus10"]) * 2.0 ** -10)
        packed = orc.q8_0_pack(w)
        assert packed.shape == (34,)
        scale = int(packed[0]) | (int(packed[1]) << 8)
        assert scale == blk["scale_bits"], blk["name"]
        np.testing.assert_array_equal(packed[2:].view(np.int8), np.array(blk["quants"], np.int8),
                                      err_msg=blk["name"])


def test_q8_0_error_bounds_and_round_trip(orc):
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    w[3, :32] = 0.0                                  # an all-zero block
    w[5, 32:64] = np.linspace(-1, 1, 32)             # amax hits both +-127
    packed = orc.q8_0_pack(w)
    assert packed.shape == (64, 8 * 34)              # 8.5 bits per weight
    back = orc.q8_0_unpack(packed, 256)
    blocks = packed.reshape(64, 8, 34)
    q = blocks[:, :, 2:].view(np.int8).astype(np.int32)
    dh = (blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
    d16 = dh.view(np.float16).astype(np.float64)
    wb = w.reshape(64, 8, 32).astype(np.float64)
    amax = np.abs(wb).max(-1)
    d32 = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    # dequant is scale * quant, exactly
    np.testing.assert_array_equal(back.reshape(64, 8, 32), (d16[..., None] * q).astype(np.float32))
    # |quant| <= 127 and the largest weight maps to +-127
    assert np.abs(q).max() <= 127
    nz = amax > 0
    assert np.all(np.abs(q).max(-1)[nz] == 127)
    # rounding error against the FP32 scale: |w/d - q| <= 1/2 (plus one f32 rounding of w/d)
    ratio = np.where(nz[..., None], wb / np.where(nz, d32, 1)[..., None], 0)
    assert np.all(np.abs(ratio - q) <= 0.5 + 1e-5)
    # full per-weight error: d/2 from rounding plus 127 * |fp16(d) - d|
    err = np.abs(back.reshape(64, 8, 32) - wb)
    bound = d32 / 2 * (1 + 1e-5) + 127 * np.abs(d16 - d32)
    assert np.all(err <= bound[..., None] + 1e-12)
    # the zero block stays zero with a zero scale
    assert dh[3, 0] == 0 and np.all(q[3, 0] == 0)


def test_q8_0_multiples_of_scale_round_trip(orc):
    rng = np.random.default_rng(3)
    for e in (-12, -9, -7, -3):
        k = rng.integers(-127, 128, size=32)
        k[0] = 127
        w = (k * 2.0 ** e).astype(np.float32)
        back = orc.q8_0_unpack(orc.q8_0_pack(w), 32)
        np.testing.assert_array_equal(back, w)


def test_affine4_hand_worked_groups(orc):
    spec = json.load(open(os.path.join(GOLDEN, "affine4_gs32_worked_example.json")))
    for grp in spec["groups"]:
        k = np.array(grp["k"], np.float64)
        assert k.shape == (32,)
        w = np.ldexp(k, grp["unit_log2"]).astype(np.float32)
        assert np.all(w.astype(np.float64) == np.ldexp(k, grp["unit_log2"]))
        packed = orc.affine4_pack(w)
        assert packed.shape == (20,), grp["name"]
        np.testing.assert_array_equal(packed[:16], np.array(grp["code_bytes"], np.uint8),
                                      err_msg=grp["name"])
        assert int(packed[16]) | (int(packed[17]) << 8) == grp["scale_bits"], grp["name"]
        assert int(packed[18]) | (int(packed[19]) << 8) == grp["bias_bits"], grp["name"]
        back = orc.affine4_unpack(packed, 32)
        for i, v in grp["dequant"]:
            assert back[i] == np.float32(v), (grp["name"], i)


def _affine4_fields(packed, rows, groups):
    g = packed.reshape(rows, groups, 20)
    codes = np.empty((rows, groups, 32), np.int64)
    codes[..., 0::2] = g[..., :16] & 0xF
    codes[..., 1::2] = g[..., :16] >> 4
    sh = (g[..., 16].astype(np.uint16) | (g[..., 17].astype(np.uint16) << 8))
    bh = (g[..., 18].astype(np.uint16) | (g[..., 19].astype(np.uint16) << 8))
    return codes, sh.view(np.float16).astype(np.float64), bh.view(np.float16).astype(np.float64)


def test_affine4_grid_rounding_bounds(orc):
    rng = np.random.default_rng(4)
    rows, n = 64, 256
    w = (rng.standard_normal((rows, n)) * 0.02).astype(np.float32)
    w[2, :32] = 0.01                                   # a constant group
    w[7, 64:96] = np.linspace(-3, 5, 32)               # a wide group
    packed = orc.affine4_pack(w)
    assert packed.shape == (rows, n // 32 * 20)        # 5.0 bits per weight
    back = orc.affine4_unpack(packed, n).reshape(rows, n // 32, 32).astype(np.float64)
    codes, s16, b16 = _affine4_fields(packed, rows, n // 32)
    wb = w.reshape(rows, n // 32, 32).astype(np.float64)
    lo, hi = wb.min(-1), wb.max(-1)
    # the stored bias and scale are the fp16 roundings of the group minimum and range / 15
    np.testing.assert_array_equal(b16, lo.astype(np.float16).astype(np.float64))
    d32 = ((hi - lo).astype(np.float32) / np.float32(15)).astype(np.float32)
    np.testing.assert_array_equal(s16, d32.astype(np.float16).astype(np.float64))
    # dequant is scale * code + bias, rounded once to FP32
    np.testing.assert_array_equal(back, (s16[..., None] * codes + b16[..., None])
                                  .astype(np.float32).astype(np.float64))
    # codes span the grid: the minimum gets 0 and the maximum 15 wherever the range is non-zero
    wide = s16 > 0
    assert np.all(codes.min(-1)[wide] == 0) and np.all(codes.max(-1)[wide] == 15)
    assert np.all(codes[~wide] == 0) and not wide[2, 0]
    # codes are monotone in the weight within a group
    order = np.argsort(wb, axis=-1, kind="stable")
    assert np.all(np.diff(np.take_along_axis(codes, order, -1), axis=-1) >= 0)
    # nearest grid point: |w - (scale * code + bias)| <= scale / 2 (plus FP32 rounding of the
    # quotient and of the dequantised value)
    grid = s16[..., None] * codes + b16[..., None]
    err = np.abs(wb - grid)
    assert np.all(err[wide] <= s16[wide][:, None] * (0.5 + 2.0 ** -18) + 1e-12)
    # a zero scale leaves every weight at the bias: off by the fp16 rounding of the minimum
    assert np.all(err[~wide] == np.abs(lo - b16)[~wide][:, None])
    assert np.all(np.abs(back - grid) <= np.abs(grid) * 2.0 ** -24)
    # the constant group comes back exactly when its value is an fp16 number
    assert np.all(back[2, 0] == np.float32(np.float16(0.01)))


def test_affine4_quantizer_keeps_its_own_output(orc):
    """A group already on an fp16 grid (minimum 0 code, maximum 15) packs to the same bytes."""
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((16, 512)) * 0.02).astype(np.float32)
    once = orc.affine4_pack(w)
    back = orc.affine4_unpack(once, 512)
    np.testing.assert_array_equal(orc.affine4_pack(back), once)
    np.testing.assert_array_equal(orc.affine4_unpack(orc.affine4_pack(back), 512), back)


def test_argmax_lowest_index_on_ties(orc):
    v = np.array([0.0, 3.0, -1.0, 3.0, 2.0], np.float32)
    assert orc.argmax(v) == 1
    assert orc.argmax(np.full(7, -2.0, np.float32)) == 0
