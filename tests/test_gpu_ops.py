"""Operator gates on the GPU: each kernel family against the oracle on the same
seeded inputs (the pages' operator tests: "Reproducing Kipp", section
"Model-backed CPU and Metal gates", --metal-operators).

- Q8_0 packing: the library's CUDA quantizer and the oracle's packer agree
  bit for bit ("Kipp Model Support", section "Quantization (Q8_0)").
- AFFINE4_GS32 packing and the fp16 copy of its groups: the CUDA quantizer
  and the oracle's packer agree bit for bit, and the fp16 copy is the fp16
  rounding of the oracle's dequantised values, bit for bit ("Kipp Model
  Support", section "Quantization (AFFINE4_GS32)").
- tcgen05 GEMM: fp16 inputs (the prefill operand type), FP32 accumulation,
  against an FP64 matmul of the same values; shapes span several tiles and ragged token counts (1, 5, 40, 83,
  200, 300) so every N tile width and the tile tail are exercised.
- Decode GEMV, BF16 and Q8_0 planes, against the oracle.
Tolerance: the products are exact in FP32 and only the K-term FP32
accumulation differs from FP64, so per element |err| <= 1e-5 * sum_k |w x|.
"""
import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q3():
    import qwen3_dense_decoder_gb300 as q3
    q3.build()
    return q3


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


def _f32(t):
    return t.float().cpu().numpy()


def test_quantizer_matches_oracle_packer_bitwise(q3, orc):
    w = _bf16((96, 4096), 1, 0.02)
    w[3, :32] = 0                                             # all-zero block
    w[4, 32:64] = torch.linspace(-1, 1, 32, device="cuda").to(torch.bfloat16)
    got = q3.quantize_q8_0(w).cpu().numpy()
    ref = orc.q8_0_pack(_f32(w))
    np.testing.assert_array_equal(got, ref)


def _affine4_edge_rows(w):
    """Edge groups: all zero, signed zeros, constant, a linear ramp, a range
    whose scale is an fp16 subnormal (codes clamp at 15), mixed signs."""
    dev = w.device
    w[3, :32] = 0
    w[4, :32] = 0
    w[4, 1:32:3] = -0.0
    w[4, 0] = -0.0
    w[5, 32:64] = 0.75
    w[6, 64:96] = torch.linspace(-1, 1, 32, device=dev).to(torch.bfloat16)
    k = torch.tensor(list(range(19)) + list(range(13)), dtype=torch.float32, device=dev)
    w[7, 96:128] = (k * 2.0 ** -24).to(torch.bfloat16)
    w[8, :32] = torch.tensor([(-1) ** i * (i + 1) for i in range(32)], dtype=torch.float32,
                             device=dev).to(torch.bfloat16)
    return w


@pytest.mark.parametrize("rows,n", [(96, 4096), (3, 7 * 32), (1, 32)])
def test_affine4_quantizer_matches_oracle_packer_bitwise(q3, orc, rows, n):
    w = _bf16((rows, n), 7, 0.02)
    if rows >= 9 and n >= 128:
        w = _affine4_edge_rows(w)
    got = q3.quantize_affine4(w).cpu().numpy()
    assert got.shape == (rows, n // 32 * 20)
    ref = orc.affine4_pack(_f32(w))
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("rows,n", [(96, 4096), (5, 9 * 32)])
def test_affine4_f16_copy_matches_oracle_dequant_bitwise(q3, orc, rows, n):
    w = _bf16((rows, n), 8, 0.02)
    if rows >= 9:
        w = _affine4_edge_rows(w)
    groups = q3.quantize_affine4(w)
    got = q3.affine4_to_f16(groups, n).cpu().numpy()
    ref = orc.affine4_unpack(groups.cpu().numpy(), n).astype(np.float16)
    np.testing.assert_array_equal(got.view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("bn", [0, 32, 64, 96, 128, 144, 160, 176, 192, 256])
@pytest.mark.parametrize("n", [1, 5, 40, 83, 200, 300])
@pytest.mark.parametrize("M,K", [(256, 64), (384, 2560), (128, 9728)])
def test_tcgen05_matmul_matches_oracle(q3, orc, n, M, K, bn):
    # bf16-valued weights (exact in fp16) so the oracle's bf16 matmul applies
    w = _bf16((M, K), 10 + n, 0.05)
    rows = (n + 255) // 256 * 256
    x = torch.randn(rows, K, generator=torch.Generator(device="cuda").manual_seed(20 + n),
                    device="cuda").to(torch.float16)
    y = q3.op_matmul(w.to(torch.float16), x, n, block_n=bn)
    torch.cuda.synchronize()
    wb = w.view(torch.int16).cpu().numpy().view(np.uint16)
    xf = _f32(x[:n])
    ref = orc.matmul(wb, 0, M, K, xf, n_threads=8)
    # tensor-core FP32 accumulation is not IEEE-ordered: allow 5e-5 of the magnitude sum
    bound = 5e-5 * (np.abs(xf.astype(np.float64)) @ np.abs(_f32(w).astype(np.float64)).T) + 1e-30
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), (err / bound).max()


@pytest.mark.parametrize("M,K", [(128, 1024), (6144, 2560), (2560, 9728), (1024, 17408)])
def test_gemv_bf16_matches_oracle(q3, orc, M, K):
    w = _bf16((M, K), 30, 0.02)
    x = torch.randn(K, generator=torch.Generator(device="cuda").manual_seed(31), device="cuda")
    y = q3.op_matvec(w, x)
    torch.cuda.synchronize()
    ref = orc.matmul(w.view(torch.int16).cpu().numpy().view(np.uint16), 0, M, K, x.cpu().numpy(),
                     n_threads=8)[0]
    bound = 1e-5 * (np.abs(_f32(w).astype(np.float64)) @ np.abs(x.cpu().numpy().astype(np.float64)))
    assert np.all(np.abs(y.cpu().numpy() - ref) <= bound)


@pytest.mark.parametrize("M,K", [(128, 1024), (4096, 4096), (4096, 12288)])
def test_gemv_q8_0_matches_oracle(q3, orc, M, K):
    w = _bf16((M, K), 40, 0.02)
    blocks = q3.quantize_q8_0(w)                              # canonical [M][K/32][34]
    b3 = blocks.view(M, K // 32, 34)
    scales = b3[:, :, 0:2].contiguous().view(torch.float16).view(M, K // 32)
    quants = b3[:, :, 2:].contiguous().view(torch.int8).view(M, K)
    x = torch.randn(K, generator=torch.Generator(device="cuda").manual_seed(41), device="cuda")
    y = q3.op_matvec(quants, x, scales)
    torch.cuda.synchronize()
    bnp = blocks.cpu().numpy()
    ref = orc.matmul(bnp, 1, M, K, x.cpu().numpy(), n_threads=8)[0]
    deq = orc.q8_0_unpack(bnp, K).astype(np.float64)
    bound = 1e-5 * (np.abs(deq) @ np.abs(x.cpu().numpy().astype(np.float64)))
    assert np.all(np.abs(y.cpu().numpy() - ref) <= bound)


@pytest.mark.parametrize("M,K", [(8, 128), (128, 1024), (6144, 2560), (2560, 9728), (1024, 17408)])
def test_gemv_affine4_matches_oracle(q3, orc, M, K):
    """The 5.0-bit AFFINE4 matvec of one-token rounds: codes dequantised in
    registers to fp16(scale * code + bias) (the values of the fp16 copy the
    tensor-core path reads, pinned bitwise above), the activation rounded to
    fp16, FP32 accumulation on mma.sync.  Against the FP64 sum of those fp16
    operands: 1e-5 of sum |w x| (the accumulation); against the oracle's
    exact AFFINE4 matmul: 2^-10 of sum |w x| (the two fp16 roundings)."""
    w = _bf16((M, K), 50, 0.02)
    if M >= 9 and K >= 128:
        w = _affine4_edge_rows(w)
    groups = q3.quantize_affine4(w)
    x = torch.randn(K, generator=torch.Generator(device="cuda").manual_seed(51), device="cuda")
    y = q3.op_matvec_affine4(groups, x, M, K).cpu().numpy().astype(np.float64)
    gnp = groups.cpu().numpy()
    deq = orc.affine4_unpack(gnp, K)
    xn = x.cpu().numpy()
    w16 = deq.astype(np.float16).astype(np.float64)
    x16 = xn.astype(np.float16).astype(np.float64)
    mag = np.abs(deq.astype(np.float64)) @ np.abs(xn.astype(np.float64)) + 1e-30
    assert np.all(np.abs(y - w16 @ x16) <= 1e-5 * (np.abs(w16) @ np.abs(x16)) + 1e-30)
    ref = orc.matmul(gnp, 2, M, K, xn, n_threads=8)[0].astype(np.float64)
    err = np.abs(y - ref)
    assert np.all(err <= 2.0 ** -10 * mag), (err / mag).max()
