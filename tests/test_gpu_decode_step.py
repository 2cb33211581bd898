"""The fused one-kernel decode step against the oracle and against the
per-operation path (same forward, "Kipp Model Support", section
"qwen3-0.6b-base"; decode gate of "What the gates check": identical argmax
and full-logit NMSE <= 1e-4 at every decode position).

The cases cover what is particular to the fused kernel: attention contexts
split over many CTAs with the new position at every offset of its 32-position
block, KV blocks taken from a permuted table, several ring slots per unit,
gate/up tiles of one and many rows (hidden 1024 .. 5120, FFN 3072 .. 17408),
Q8_0 projection planes, a bad token, and one launch per step.
"""
import numpy as np
import pytest
import torch

import synthetic
from helpers import NMSE_BOUND, Pair, check_row, make_shape

pytestmark = pytest.mark.gpu

TINY = make_shape("tiny")


def _decode(pair, g, o, tok, n, tag):
    checks = []
    for step in range(n):
        got, ref, am = pair.eval(g, o, [tok])
        c = check_row(got, ref, tag)
        assert am == c.argmax_gpu, (tag, step)
        assert c.ok, (tag, step, c)
        checks.append(c)
        tok = c.argmax_ref
    return checks, tok


@pytest.fixture(scope="module")
def long_pair():
    return Pair(TINY, seed=111, max_ctx=2048, max_round_tokens=256, n_blocks=80)


def test_fused_step_is_the_default_and_one_launch(long_pair):
    m = long_pair.model
    assert m.fused_decode
    g, o = long_pair.sessions()
    prompt = synthetic.make_tokens(20, TINY.vocab, seed=40)
    got, ref, _ = long_pair.eval(g, o, prompt)
    assert check_row(got, ref).ok
    before = m.launch_count
    _decode(long_pair, g, o, int(np.argmax(ref)), 3, "launches")
    assert m.launch_count - before == 3
    g.close()


def test_fused_step_long_split_context_permuted(long_pair):
    # 1,500-token context over 47 blocks of a permuted table: attention units
    # span several ring slots, and 40 decode steps move the new position across
    # a block edge (1,504 and 1,536)
    perm = synthetic.make_block_permutation(80, seed=41)
    g, o = long_pair.sessions(table=perm[:50])
    prompt = synthetic.make_tokens(1500, TINY.vocab, seed=42)
    for a in range(0, 1500, 256):
        got, ref, _ = long_pair.eval(g, o, prompt[a:a + 256])
        assert check_row(got, ref).ok, a
    checks, _ = _decode(long_pair, g, o, int(np.argmax(ref)), 40, "tiny-long")
    assert max(c.nmse for c in checks) <= NMSE_BOUND
    assert g.pos == 1540
    g.close()


def test_fused_equals_per_operation_path(long_pair):
    # the same session state decoded by both paths: both within the bound of
    # the oracle, and close to each other (they differ in summation order only)
    m = long_pair.model
    prompt = synthetic.make_tokens(100, TINY.vocab, seed=43)
    outs = {}
    for fused in (True, False):
        m.set_fused_decode(fused)
        g, o = long_pair.sessions()
        got, ref, _ = long_pair.eval(g, o, prompt)
        checks, _ = _decode(long_pair, g, o, int(np.argmax(ref)), 6, f"fused={fused}")
        outs[fused] = long_pair.logits[0].cpu().numpy().copy()
        g.close()
    m.set_fused_decode(True)
    assert check_row(outs[True], outs[False]).nmse <= 1e-8


def test_fused_step_first_token_is_a_decode_round(long_pair):
    # a one-token round at position 0: the whole context is the new position
    g, o = long_pair.sessions()
    checks, _ = _decode(long_pair, g, o, 7, 33, "from-zero")
    assert g.pos == 33
    g.close()


def test_fused_step_bad_token_is_a_device_check():
    import qwen3_dense_decoder_gb300 as q3
    pair = Pair(TINY.replace(n_layers=1), seed=44, max_ctx=64, max_round_tokens=32, n_blocks=4)
    assert pair.model.fused_decode
    g = pair.pool.session()
    g.eval(torch.tensor([1, 2], dtype=torch.int32, device="cuda"), pair.logits[0])
    pair.model.sync()
    g.eval(torch.tensor([TINY.vocab], dtype=torch.int32, device="cuda"), pair.logits[0])
    with pytest.raises(q3.Q3Error) as e:
        pair.model.sync()
    assert e.value.code == -7


def test_fused_step_q8_0_planes():
    shape = make_shape("8b-q8_0", n_layers=2)
    pair = Pair(shape, seed=45, max_ctx=256, max_round_tokens=64, n_blocks=8)
    assert pair.model.fused_decode
    g, o = pair.sessions(table=synthetic.make_block_permutation(8, seed=46)[:4])
    prompt = synthetic.make_tokens(40, shape.vocab, seed=47)
    got, ref, _ = pair.eval(g, o, prompt)
    assert check_row(got, ref).ok
    _decode(pair, g, o, int(np.argmax(ref)), 6, "8b-q8_0")


def test_fused_step_14b_shape_two_layers():
    # hidden 5120 (3 ring slots), FFN 17408: one down-projection row per slot
    shape = make_shape("14b", n_layers=2)
    pair = Pair(shape, seed=48, max_ctx=128, max_round_tokens=64, n_blocks=8)
    assert pair.model.fused_decode
    g, o = pair.sessions(table=synthetic.make_block_permutation(8, seed=49)[:3])
    prompt = synthetic.make_tokens(33, shape.vocab, seed=50)
    got, ref, _ = pair.eval(g, o, prompt)
    assert check_row(got, ref).ok
    _decode(pair, g, o, int(np.argmax(ref)), 4, "14b")
