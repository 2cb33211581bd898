"""The projection-GEMM planner (host logic, no GPU): the token-tile widths and
K-split counts a model's rounds use, the plans the benchmark's workloads run
on, and which prefill rounds apply the q/k head norm, RoPE and K/V append in
the QKV GEMM's epilogue (no K split) rather than in the separate kernel."""
import pytest

import synthetic

WIDTHS = (32, 64, 96, 128, 144, 160, 176, 192, 256)
WS_FLOATS = 32 << 20


@pytest.fixture(scope="module")
def q3():
    import qwen3_dense_decoder_gb300 as q3
    q3.build()
    return q3


def qkv_rows(s):
    return (s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim


def test_plans_of_the_benchmark_workloads(q3):
    s = synthetic.SHAPES["4b"]
    H, F, Q = s.hidden, s.ffn, s.n_q_heads * s.head_dim
    # a 2,048-token prefill round
    assert q3.gemm_plan(qkv_rows(s), 2048, H) == (256, 1)
    assert q3.gemm_plan(H, 2048, Q) == (144, 1)          # O: 20 x 15 = 300 tiles, 1.97 waves
    assert q3.gemm_plan(H, 2048, F) == (144, 1)          # down
    assert q3.gemm_plan(2 * F, 2048, H) == (256, 1)      # gate/up rows paired
    # a batch-32 decode round: weight-streaming GEMMs whose tiles do not fill the SMs
    assert q3.gemm_plan(qkv_rows(s), 32, H) == (32, 3)
    assert q3.gemm_plan(H, 32, Q) == (32, 7)
    assert q3.gemm_plan(H, 32, F) == (32, 7)


@pytest.mark.parametrize("M,K", [(4096, 1024), (6144, 2560), (2560, 4096), (2560, 9728), (19456, 2560),
                                 (7168, 5120), (5120, 17408)])
def test_plan_invariants(q3, M, K):
    for N in (1, 2, 7, 31, 32, 33, 64, 65, 100, 128, 129, 300, 777, 1024, 2048):
        bn, ks = q3.gemm_plan(M, N, K)
        assert bn in WIDTHS
        # never wider than the rows need (tiles of 32, 64 or 128 for short rounds)
        assert bn <= (32 if N <= 32 else 64 if N <= 64 else 128 if N <= 128 else 256)
        assert 1 <= ks <= 8
        if ks > 1:
            assert K // 64 // ks >= 4                     # each split keeps 4 k-blocks
            assert ks * N * M <= WS_FLOATS                # the partials fit the workspace
        tiles = (M // 128) * -(-N // bn)
        if tiles >= 152:                                  # tiles fill the SMs: 1, 2 or 4 splits
            assert ks in (1, 2, 4)


@pytest.mark.parametrize("key", sorted(synthetic.SHAPES))
def test_prefill_rounds_that_take_the_head_epilogue(q3, key):
    """Rounds whose QKV plan splits K are a prefix of short rounds; every
    round of 64 tokens or more takes the head epilogue."""
    s = synthetic.SHAPES[key]
    split = [T for T in range(1, 2049) if q3.gemm_plan(qkv_rows(s), T, s.hidden)[1] > 1]
    assert split == list(range(1, len(split) + 1))
    assert 0 < len(split) < 64


def test_tiny_rounds_of_the_gpu_head_epilogue_test(q3):
    s = synthetic.SHAPES["tiny"]
    assert q3.gemm_plan(qkv_rows(s), 20, s.hidden)[1] > 1       # the separate kernel
    assert q3.gemm_plan(qkv_rows(s), 70, s.hidden) == (32, 1)    # 32-token tiles, 6-token tail
    assert q3.gemm_plan(qkv_rows(s), 170, s.hidden) == (64, 1)   # 64-token tiles, 42-token tail


def test_bad_arguments_are_rejected(q3):
    big = (1 << 18) + 128
    for M, N, K in ((100, 32, 64), (128, 0, 64), (128, 32, 100), (0, 32, 64), (big, 32, 64), (128, big, 64),
                    (128, 32, (1 << 18) + 64)):
        with pytest.raises(q3.Q3Error):
            q3.gemm_plan(M, N, K)
