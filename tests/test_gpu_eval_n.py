"""Multi-logit evaluation (q3_session_eval_n) against the oracle's every-row
logits ("Kipp Roadmap", status v0.0.2: multi-logit evaluation,
kipp_session_eval_n; decode gate of "Kipp Model Support", section "What the
gates check": identical argmax and full-logit NMSE <= 1e-4 per row).

Cases: every row of a prompt scored, a suffix of the rows, one row (equal to
q3_session_eval bitwise), and a prompt longer than max_round_tokens whose
scored rows straddle two rounds.
"""
import numpy as np
import pytest
import torch

import synthetic
from helpers import Pair, check_row, make_shape

pytestmark = pytest.mark.gpu

TINY = make_shape("tiny")


@pytest.fixture(scope="module")
def pair():
    return Pair(TINY, seed=121, max_ctx=512, max_round_tokens=64, n_blocks=64)


def _scored(pair, tokens, n_logits, table=None):
    g, o = pair.sessions(table=table)
    V = TINY.vocab
    lg = torch.empty(n_logits, V, dtype=torch.float32, device="cuda")
    am = torch.empty(n_logits, dtype=torch.int32, device="cuda")
    g.eval_n(torch.tensor(tokens, dtype=torch.int32, device="cuda"), n_logits, lg, am)
    pair.model.sync()
    ref = o.eval(tokens, all_rows=True)[-n_logits:]
    got = lg.cpu().numpy()
    amx = am.cpu().numpy()
    for i in range(n_logits):
        c = check_row(got[i], ref[i], f"eval_n/{len(tokens)}/{n_logits}")
        assert c.ok, (i, c)
        assert amx[i] == c.argmax_gpu, i
    assert g.pos == len(tokens)
    g.close()
    return got


def test_every_prompt_row_scored(pair):
    _scored(pair, synthetic.make_tokens(50, TINY.vocab, seed=60), 50,
            table=synthetic.make_block_permutation(64, seed=61)[:4])


def test_suffix_of_rows_scored(pair):
    _scored(pair, synthetic.make_tokens(45, TINY.vocab, seed=62), 17)


def test_scored_rows_straddle_two_rounds(pair):
    # 150 tokens in rounds of 64, 64, 22: the last 40 rows start inside the second round
    _scored(pair, synthetic.make_tokens(150, TINY.vocab, seed=63), 40)


def test_one_scored_row_equals_eval(pair):
    toks = synthetic.make_tokens(30, TINY.vocab, seed=64)
    got = _scored(pair, toks, 1)
    g, _ = pair.sessions()
    g.eval(torch.tensor(toks, dtype=torch.int32, device="cuda"), pair.logits[0])
    pair.model.sync()
    np.testing.assert_array_equal(got[0], pair.logits[0].cpu().numpy())
    g.close()


def test_bad_logit_count_is_rejected(pair):
    import qwen3_dense_decoder_gb300 as q3
    g, _ = pair.sessions()
    lg = torch.empty(8, TINY.vocab, dtype=torch.float32, device="cuda")
    with pytest.raises(q3.Q3Error):
        g.eval_n(torch.tensor([1, 2, 3], dtype=torch.int32, device="cuda"), 4, lg)
    with pytest.raises(q3.Q3Error):
        g.eval_n(torch.tensor([1, 2, 3], dtype=torch.int32, device="cuda"), 0, lg)
    assert g.pos == 0
    g.close()
