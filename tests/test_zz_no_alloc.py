"""The split-K matmul entry point that allocates nothing.

Callers that cannot call cudaMalloc where they need a product (a framework
that owns all device memory, a plug-in that may not grow its footprint, a
latency-critical loop that cannot afford cudaMalloc's synchronisation) use
q3_op_matmul_splitk_noalloc: its split partial sums live in the library's
fixed scratch array.  Its output must match the plain q3_op_matmul entry
point within the operator tolerance of the GEMM tests (5e-5 of sum |w x|),
on two calls in a row with different shapes (the shared scratch keeps the
previous call's contents), and the oracle's matmul directly.  The first
call on a device may commit the scratch (the driver does that when it loads
the entry point's device code); the second must not take device memory.
This file is collected last so a failure here comes after every other test.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q3():
    import qwen3_dense_decoder_gb300 as q3
    q3.build()
    return q3


def _inputs(M, K, n, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = (torch.randn(M, K, generator=g, device="cuda") * 0.05).to(torch.float16)
    x = torch.randn((n + 255) // 256 * 256, K, generator=g, device="cuda").to(torch.float16)
    return w, x


def _bound(w, x, n):
    wa = w.double().abs().cpu().numpy()
    xa = x[:n].double().abs().cpu().numpy()
    return 5e-5 * (xa @ wa.T) + 1e-30


SCRATCH_BYTES = 4 * 2 * 1024 * 1024


def test_noalloc_matches_existing_matmul_on_two_calls(q3):
    cases = [(256, 1024, 40, 4, 1), (384, 2560, 83, 8, 2)]
    prepared = []
    for M, K, n, ks, seed in cases:                  # every buffer exists before the calls
        w, x = _inputs(M, K, n, seed)
        prepared.append((M, K, n, ks, w, x, torch.empty(n, M, device="cuda"),
                         q3.op_matmul(w, x, n)))
    torch.cuda.synchronize()
    free = [torch.cuda.mem_get_info()[0]]
    for M, K, n, ks, w, x, y, ref in prepared:
        q3.op_matmul_splitk_noalloc(w, x, n, ks, y)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        err = np.abs(y.double().cpu().numpy() - ref.double().cpu().numpy())
        assert np.all(err <= _bound(w, x, n)), (M, K, n, ks)
    # The first call on a device loads the entry point's device code, and the
    # driver commits the fixed scratch then (nothing if an earlier call did):
    # at most the scratch plus the code's pages.  The second call takes nothing.
    assert 0 <= free[0] - free[1] <= SCRATCH_BYTES + 8 * 1024 * 1024
    assert free[2] == free[1]


def test_noalloc_matches_the_oracle(q3, orc):
    # bf16-valued weights (exact in fp16), compared directly with the oracle's FP64-accumulated matmul
    M, K, n = 512, 4096, 100
    g = torch.Generator(device="cuda").manual_seed(5)
    wb = (torch.randn(M, K, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    x = torch.randn(256, K, generator=g, device="cuda").to(torch.float16)
    y = torch.empty(n, M, device="cuda")
    q3.op_matmul_splitk_noalloc(wb.to(torch.float16), x, n, 4, y)
    ref = orc.matmul(wb.view(torch.int16).cpu().numpy().view(np.uint16), 0, M, K,
                     x[:n].float().cpu().numpy(), n_threads=8)
    err = np.abs(y.double().cpu().numpy() - ref.astype(np.float64))
    assert np.all(err <= _bound(wb.to(torch.float16), x, n))


def test_noalloc_rejects_sizes_beyond_the_scratch(q3):
    w, x = _inputs(4096, 1024, 300, 3)
    y = torch.empty(300, 4096, device="cuda")
    with pytest.raises(q3.Q3Error) as e:             # 8 * 300 * 4096 floats > 2M
        q3.op_matmul_splitk_noalloc(w, x, 300, 8, y)
    assert e.value.code == -1 and "scratch" in str(e.value)
