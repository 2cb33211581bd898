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


PART_ROWS = 2 * 8 * 152 + 64      # (row, split) pairs the attention's partial buffers hold


def test_attention_plans_of_the_benchmark_workloads(q3):
    assert q3.attention_plan(8, 32, 2300) == 3        # batch-32 decode, longest context ~2,300
    assert q3.attention_plan(8, 1, 2176) == 17        # one session at ~2,176 (the per-operation path)
    assert q3.attention_plan(8, 8, 16448) == 17       # 8 sessions at ~16k (14B long-context decode)


@pytest.mark.parametrize("n_kv", [4, 8])
def test_attention_plan_rule(q3, n_kv):
    for T in (1, 2, 8, 32, 64, 151, 152, 200):
        for ctx in (1, 31, 32, 33, 100, 1000, 2176, 4096, 16448, 40000):
            s = q3.attention_plan(n_kv, T, ctx)
            nblk = -(-ctx // 32)
            rows = T * n_kv
            assert 1 <= s <= min(nblk, 128)
            assert s == 1 or T * s <= PART_ROWS
            if rows >= 8 * 152:
                assert s == 1                         # enough rows: no splitting
                continue
            if rows * -(-nblk // 4) <= 3 * 152 and T * min(-(-nblk // 4), 128) <= PART_ROWS:
                assert s == min(-(-nblk // 4), 128, nblk)   # one block per warp fits a wave
            else:
                assert s == 1 or -(-nblk // s) <= 8 * 4 or s == 128 or T * (s + 1) > PART_ROWS


def test_attention_plan_bad_arguments(q3):
    for args in ((0, 1, 100), (8, 0, 100), (8, 1, 0), (65, 1, 100), (8, (1 << 16) + 1, 100)):
        with pytest.raises(q3.Q3Error):
            q3.attention_plan(*args)
