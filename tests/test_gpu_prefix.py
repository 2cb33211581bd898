"""Content-addressed prefix sharing on the CUDA path ("Kipp Roadmap", status
v0.0.3: pooled sessions share one model-owned slab through a
content-addressed 32-token block pool, publish-at-finish, memcmp-verified).

A position's K/V depends only on the tokens up to it, so a session that
attaches a published chain and evaluates the rest of its prompt must give
the logits of a fresh session that evaluates the whole prompt in the same
rounds, bit for bit (the kernels are deterministic and a round's plan depends
only on the round).  Each case also passes the usual gate against the
oracle's unshared evaluation, and the attached counts equal the oracle's
under the same publish / attach sequence.  Cases: a partial match, whole-
prompt matches (one token always stays to evaluate), forced hash collisions
(one bucket), deduplicated publishing, truncation into a shared block (a
copy first; the published block stays intact), eviction under pressure (held
blocks are never evicted), and argument errors.
"""
import numpy as np
import pytest
import torch

import synthetic
from helpers import check_row, make_shape

pytestmark = pytest.mark.gpu

TINY = make_shape("tiny")


class Side:
    """A GPU model and pool with the prefix index on, and the oracle's twin."""

    def __init__(self, hash_bits=16, n_blocks=64):
        import oracle
        import qwen3_dense_decoder_gb300 as q3
        self.q3 = q3
        self.w = synthetic.make_weights(TINY, seed=77, device="cuda")
        self.model = q3.Model(TINY, q3.device_weights(TINY, self.w), max_ctx=512, max_round_tokens=256)
        self.pool = self.model.pool(n_blocks, 16)
        self.pool.enable_prefix(hash_bits)
        self.orc = oracle.Model(TINY, self.w)
        self.opool = self.orc.pool(n_blocks)
        self.opool.enable_prefix(hash_bits)
        self.logits = torch.empty(TINY.vocab, dtype=torch.float32, device="cuda")

    def run(self, g, toks):
        g.eval(torch.tensor(np.asarray(toks, np.int32), device="cuda"), self.logits)
        self.model.sync()
        return self.logits.cpu().numpy().copy()

    def rounds(self, g, toks, cuts):
        """Evaluate toks in rounds ending at each cut; the last round's logits."""
        a, out = 0, None
        for b in cuts:
            out = self.run(g, toks[a:b])
            a = b
        return out

    def oracle_fresh(self, toks):
        return self.orc.session(max_ctx=512).eval(toks)

    def osession(self):
        return self.orc.session(pool=self.opool, max_ctx=512)


def _prompt(n, seed):
    return synthetic.make_tokens(n, TINY.vocab, seed=seed)


def test_attach_then_evaluate_equals_fresh_bitwise():
    sd = Side()
    P = _prompt(200, 1)
    a, oa = sd.pool.session(), sd.osession()
    sd.rounds(a, P, [128, 200])
    oa.eval(P)
    assert a.publish(P) == oa.publish() == 6                   # positions 0..191
    P2 = np.concatenate([P[:150], _prompt(40, 2)])
    b, ob = sd.pool.session(), sd.osession()
    n = b.attach_prefix(P2)
    assert n == ob.attach_prefix(P2) == 128                     # block 4 differs at 150
    assert b.pos == 128
    got = sd.run(b, P2[n:])
    f = sd.pool.session()                                       # fresh, the same rounds
    want = sd.rounds(f, P2, [128, 190])
    np.testing.assert_array_equal(got, want)
    c = check_row(got, sd.oracle_fresh(P2), "prefix/attach")
    assert c.ok, c
    seq = P2.copy()
    for t in _prompt(4, 3):                                     # decoding on from the shared prefix
        seq = np.append(seq, t)
        g1, g2 = sd.run(b, [t]), sd.run(f, [t])
        np.testing.assert_array_equal(g1, g2)
        c = check_row(g1, sd.oracle_fresh(seq), "prefix/decode")
        assert c.ok, c


@pytest.mark.parametrize("n", [96, 97, 33, 32, 1])
def test_a_whole_prompt_match_leaves_one_token(n):
    sd = Side()
    P = _prompt(128, 4)
    got = (n - 1) // 32 * 32
    a = sd.pool.session()
    sd.rounds(a, P, [got, 128] if got else [128])      # positions < got in a round of got rows
    a.publish(P)
    s = sd.pool.session()
    assert s.attach_prefix(P[:n]) == got
    assert got == (n - 1) // 32 * 32
    out = sd.run(s, P[got:n])
    f = sd.pool.session()
    np.testing.assert_array_equal(out, sd.rounds(f, P, [got, n] if got else [n]))


def test_collisions_dedup_and_truncation_into_a_shared_block():
    sd = Side(hash_bits=0)                                      # one bucket: every lookup meets every block
    P = _prompt(100, 4)
    variant = P.copy()
    variant[40] = (variant[40] + 1) % TINY.vocab               # same block 0, another block 1
    a, oa = sd.pool.session(), sd.osession()
    sd.rounds(a, P, [64, 96, 100])
    oa.eval(P)
    assert a.publish(P) == oa.publish() == 3
    v, ov = sd.pool.session(), sd.osession()
    sd.rounds(v, variant, [64, 100])
    ov.eval(variant)
    assert v.publish(variant) == ov.publish() == 2             # block 0 shared, 1 and 2 its own
    b, ob = sd.pool.session(), sd.osession()
    sd.run(b, P)
    ob.eval(P)
    assert b.publish(P) == ob.publish() == 0                   # switched to a's blocks
    probe = variant.copy()
    probe[70] = (probe[70] + 7) % TINY.vocab                   # blocks 0, 1 of the variant
    s, os_ = sd.pool.session(), sd.osession()
    assert s.attach_prefix(probe) == os_.attach_prefix(probe) == 64
    f = sd.pool.session()
    np.testing.assert_array_equal(sd.run(s, probe[64:]), sd.rounds(f, probe, [64, 100]))
    c = sd.pool.session()
    assert c.attach_prefix(P) == 96
    c.truncate(40)                                              # inside shared block 1: copied first
    new = _prompt(30, 5)
    seq = np.concatenate([P[:40], new])
    r = check_row(sd.run(c, new), sd.oracle_fresh(seq), "prefix/truncate")
    assert r.ok, r
    d = sd.pool.session()                                       # the published blocks are intact
    assert d.attach_prefix(P) == 96
    f2 = sd.pool.session()
    np.testing.assert_array_equal(sd.run(d, P[96:]), sd.rounds(f2, P, [64, 96, 100]))


def test_eviction_spares_held_blocks():
    sd = Side(n_blocks=8)
    P, Q = _prompt(96, 6), _prompt(96, 7)
    a = sd.pool.session()
    sd.rounds(a, P, [64, 96])                                   # blocks 0, 1, 2
    a.publish(P)
    a.close()                                                   # held by the index alone
    h = sd.pool.session()
    assert h.attach_prefix(P) == 64                             # h holds blocks 0 and 1
    b = sd.pool.session()
    sd.run(b, Q)                                                # blocks 3, 4, 5
    b.publish(Q)
    b.close()
    out = sd.run(h, P[64:96])                                   # block 6; block 7 stays free
    f = sd.pool.session()
    # a fresh evaluation needs 3 blocks: block 7, then the published leaves
    # held by the index alone, oldest first (P's block 2, then Q's block 5);
    # h's blocks 0 and 1 are never candidates
    np.testing.assert_array_equal(out, sd.rounds(f, P, [64, 96]))
    f.close()
    g = sd.pool.session()
    with pytest.raises(sd.q3.Q3Error) as e:                     # every block held or a parent
        sd.run(g, _prompt(8 * 32, 8))
    assert e.value.code == -4


def test_prefix_argument_errors():
    sd = Side()
    s = sd.pool.session()
    with pytest.raises(sd.q3.Q3Error):
        sd.pool.enable_prefix(16)                               # only once
    with pytest.raises(sd.q3.Q3Error):
        s.publish(_prompt(3, 9))                                # tokens must cover the positions
    sd.run(s, _prompt(40, 9))
    with pytest.raises(sd.q3.Q3Error):
        s.attach_prefix(_prompt(40, 9))                         # only on an empty session
    t = sd.pool.session()
    t.set_block_table([60, 61])
    with pytest.raises(sd.q3.Q3Error):
        t.attach_prefix(_prompt(40, 9))                         # not with a fixed table
