"""Operator gate of the prefill attention: the tcgen05 kernel and the mma.sync
kernel against the oracle's GQA attention on the same seeded inputs
("Kipp Roadmap", status v0.0.3: flash-attention prefill kernel; "Kipp Model
Support", section "qwen3-0.6b-base": BF16 K/V in 32-position blocks).

Each row t of a round (position pos0 + t) attends to positions 0 .. pos0 + t
of its session, read through a seeded permuted block table.  The cases span
query-head groups of 1, 2, 4 and 5 (the 14B shape leaves 3 of 128 tile rows
unused), rounds of one row, ragged tiles, context before the round, and
rounds with more (tile, KV head) items than CTAs, so a CTA walks several
items back to back.

Tolerance: Q and the K/V values are exact in fp16; the kernels round the
softmax weights to fp16 (relative 2^-11, lazily rescaled so they never pass
256) and the output to fp16.  Per element
|err| <= 2^-9 max|V| + 2^-10 |ref|.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def q3():
    import qwen3_dense_decoder_gb300 as q3
    q3.build()
    return q3


def _case(n_q, n_kv, pos0, T, seed):
    ctx = pos0 + T
    nblk = (ctx + 31) // 32
    n_blocks = nblk + 5
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(T, n_q, D, generator=g, device="cuda").to(torch.float16)
    kv = torch.randn(n_blocks, 2, n_kv, 32, D, generator=g, device="cuda").to(torch.bfloat16)
    table = torch.from_numpy(np.random.default_rng(seed).permutation(n_blocks)[:nblk].astype(np.int32)).cuda()
    return q, kv, table


def _reference(orc, q, kv, table, pos0, n_kv):
    T, n_q, _ = q.shape
    ctx = pos0 + T
    bits = kv.view(torch.int16).cpu().numpy().view(np.uint16)
    tab = table.cpu().numpy()
    j = np.arange(ctx)
    K = bits[tab[j // 32], 0, :, j % 32, :]                  # [ctx, n_kv, D]
    V = bits[tab[j // 32], 1, :, j % 32, :]
    qf = q.float().cpu().numpy()
    ref = np.empty((T, n_q * D), np.float32)
    for t in range(T):
        n = pos0 + t + 1
        ref[t] = orc.gqa_attend(qf[t], K[:n], V[:n], n_q, n_kv, D).reshape(-1)
    vmax = np.abs(orc.bf16_to_f32(V)).max()
    return ref, vmax


CASES = [
    (32, 8, 0, 1), (32, 8, 0, 37), (32, 8, 0, 300), (32, 8, 200, 83), (32, 8, 1000, 130),
    (32, 8, 0, 1200),                      # 304 items: two per CTA
    (40, 8, 0, 260), (40, 8, 77, 50),      # G = 5
    (16, 8, 0, 300), (16, 8, 31, 97),      # G = 2
    (8, 8, 0, 200),                        # G = 1
    (40, 8, 10000, 64),                    # a late chunk of a long prefill (the 14B shape's heads)
]


@pytest.mark.parametrize("use_tc", [True, False])
@pytest.mark.parametrize("n_q,n_kv,pos0,T", CASES)
def test_prefill_attention_matches_oracle(q3, orc, n_q, n_kv, pos0, T, use_tc):
    q, kv, table = _case(n_q, n_kv, pos0, T, seed=1000 + 7 * T + pos0 + n_q)
    out = q3.op_prefill_attention(q, kv, table, pos0, n_kv, use_tc=use_tc)
    ref, vmax = _reference(orc, q, kv, table, pos0, n_kv)
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    bound = 2.0 ** -9 * vmax + 2.0 ** -10 * np.abs(ref)
    err = np.abs(got - ref)
    assert np.all(err <= bound), (float((err / bound).max()), np.unravel_index(np.argmax(err / bound), err.shape))


def test_prefill_attention_tc_matches_mma_sync(q3):
    # the two kernels differ in summation order and in where P is rounded only
    q, kv, table = _case(32, 8, 300, 700, seed=77)
    a = q3.op_prefill_attention(q, kv, table, 300, 8, use_tc=True).float()
    b = q3.op_prefill_attention(q, kv, table, 300, 8, use_tc=False).float()
    nmse = float(((a - b) ** 2).sum() / (b ** 2).sum())
    assert nmse <= 4e-6, nmse


@pytest.mark.parametrize("use_tc", [True, False])
def test_prefill_attention_bad_block_is_a_device_check(q3, use_tc):
    q, kv, table = _case(32, 8, 0, 70, seed=5)
    table[1] = kv.shape[0]                                   # one past the pool
    with pytest.raises(q3.Q3Error) as e:
        q3.op_prefill_attention(q, kv, table, 0, 8, use_tc=use_tc)
    assert e.value.code == -7
    status = int(str(e.value).rsplit("0x", 1)[1], 16)
    assert status & 0x2                                       # Q3_STATUS_BLOCK_RANGE
