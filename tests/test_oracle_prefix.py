"""Pins of the oracle's content-addressed prefix sharing ("Kipp Roadmap",
status v0.0.3: pooled sessions share one model-owned slab through a
content-addressed 32-token block pool, publish-at-finish, memcmp-verified).

A position's K/V depends only on the tokens up to it, so a session that
attaches a published chain and evaluates the rest of its prompt must give
logits bitwise equal to evaluating the whole prompt; the cases below hold
that against plain sessions, under forced hash collisions, after
deduplication, under eviction pressure and after a truncation into a shared
block (which must leave the published copy untouched).
"""
import numpy as np
import pytest

from synthetic import Shape, make_tokens, make_weights

TINY = Shape("oracle-tiny", 2, 64, 4, 2, 16, 96, 128, True, rope_theta=1e4)


@pytest.fixture(scope="module")
def model(orc):
    return orc.Model(TINY, make_weights(TINY, seed=7), n_threads=2)


def _fresh(model, toks):
    return model.session(max_ctx=256).eval(toks, all_rows=True)


def _prompt(n, seed):
    return make_tokens(n, TINY.vocab, seed=seed)


def _pool(model, n_blocks=64, hash_bits=16):
    pool = model.pool(n_blocks)
    pool.enable_prefix(hash_bits)
    return pool


def _publish(model, pool, toks):
    s = model.session(pool=pool, max_ctx=256)
    s.eval(toks)
    return s, s.publish()


def test_attached_prefix_equals_recompute(model):
    pool = _pool(model)
    P = _prompt(100, 1)
    a, n = _publish(model, pool, P)
    assert n == 3                                    # positions 0..95; 96..99 stay private
    P2 = np.concatenate([P[:70], _prompt(30, 2)])
    b = model.session(pool=pool, max_ctx=256)
    assert b.attach_prefix(P2) == 64                 # blocks 0 and 1; block 2 differs at 70
    assert b.pos == 64
    ref = _fresh(model, P2)
    np.testing.assert_array_equal(b.eval(P2[64:], all_rows=True), ref[64:])
    # decoding on from the attached prefix matches too
    f = model.session(max_ctx=256)
    f.eval(P2)
    for t in _prompt(5, 3):
        np.testing.assert_array_equal(b.eval(np.array([t], np.int32)), f.eval(np.array([t], np.int32)))


@pytest.mark.parametrize("n", [96, 97, 33, 32, 1])
def test_a_whole_prompt_match_leaves_one_token(model, n):
    pool = _pool(model)
    P = _prompt(128, 4)
    _publish(model, pool, P)
    s = model.session(pool=pool, max_ctx=256)
    got = s.attach_prefix(P[:n])
    assert got == (n - 1) // 32 * 32
    np.testing.assert_array_equal(s.eval(P[got:n], all_rows=True), _fresh(model, P[:n])[got:])


def test_forced_collisions_are_resolved_by_comparing_tokens(model):
    pool = _pool(model, hash_bits=0)                 # one bucket: every lookup meets every block
    base = _prompt(96, 5)
    variants = []
    for k in range(3):                               # same block 0, different block 1
        v = base.copy()
        v[40] = (v[40] + 1 + k) % TINY.vocab
        variants.append(v)
    swapped = base.copy()                            # same block 1 tokens, different block 0
    swapped[3] = (swapped[3] + 1) % TINY.vocab
    for v in [base] + variants + [swapped]:
        _publish(model, pool, v)
    probe = base.copy()
    probe[70] = (probe[70] + 7) % TINY.vocab         # blocks 0, 1 as base; block 2 differs
    s = model.session(pool=pool, max_ctx=256)
    assert s.attach_prefix(probe) == 64
    np.testing.assert_array_equal(s.eval(probe[64:], all_rows=True), _fresh(model, probe)[64:])
    # a prompt whose block 1 matches a published block 1 under another block 0 attaches nothing more
    other = swapped.copy()
    other[0] = (other[0] + 3) % TINY.vocab
    s2 = model.session(pool=pool, max_ctx=256)
    assert s2.attach_prefix(other) == 0
    # and the variant chains attach exactly their own blocks
    for v in variants:
        s3 = model.session(pool=pool, max_ctx=256)
        assert s3.attach_prefix(v) == 64
        np.testing.assert_array_equal(s3.eval(v[64:], all_rows=True), _fresh(model, v)[64:])


def test_a_block_is_matched_under_its_own_parent_only(model):
    """[A, D] must not take D published after C: same tokens, another prefix, other K/V."""
    pool = _pool(model, hash_bits=0)
    A, B, Cb, D = (_prompt(32, 40 + k) for k in range(4))
    _publish(model, pool, np.concatenate([A, B]))
    _publish(model, pool, np.concatenate([Cb, D]))
    probe = np.concatenate([A, D, _prompt(5, 44)])
    s = model.session(pool=pool, max_ctx=256)
    assert s.attach_prefix(probe) == 32
    np.testing.assert_array_equal(s.eval(probe[32:], all_rows=True), _fresh(model, probe)[32:])


def test_publishing_an_equal_chain_shares_the_first_copy(model):
    pool = _pool(model, n_blocks=32)
    P = _prompt(64, 6)
    a = model.session(pool=pool, max_ctx=256)
    a.eval(P)
    b = model.session(pool=pool, max_ctx=256)
    b.eval(P)
    assert pool.free_blocks == 32 - 4
    assert a.publish() == 2
    assert b.publish() == 0                          # b now holds a's blocks; its own are free
    assert pool.free_blocks == 32 - 2
    del a, b
    assert pool.free_blocks == 32 - 2                # the index keeps the published pair
    c = model.session(pool=pool, max_ctx=256)
    assert c.attach_prefix(np.concatenate([P, _prompt(3, 7)])) == 64


def test_eviction_spares_blocks_a_session_holds(model):
    pool = _pool(model, n_blocks=8)
    P = _prompt(64, 8)
    a, _ = _publish(model, pool, P)
    del a                                           # only the index holds P's two blocks
    x = model.session(pool=pool, max_ctx=256)
    assert x.attach_prefix(np.concatenate([P, _prompt(1, 9)])) == 64
    # fill the pool with other published prompts until blocks must be evicted
    for k in range(6):
        s, n = _publish(model, pool, _prompt(64, 100 + k))
        assert n == 2
        del s
    # x's attached blocks were never evicted: its continuation equals a recompute
    tail = _prompt(20, 10)
    full = np.concatenate([P, tail])
    np.testing.assert_array_equal(x.eval(tail, all_rows=True), _fresh(model, full)[64:])
    # with every block held by live sessions, a new round cannot get one
    live = [x]
    while pool.free_blocks:
        s = model.session(pool=pool, max_ctx=256)
        s.eval(_prompt(32, 200 + len(live)))
        live.append(s)
    with pytest.raises(RuntimeError):
        for k in range(8):                           # evicts the last published leaves, then fails
            t = model.session(pool=pool, max_ctx=256)
            t.eval(_prompt(32, 300 + k))
            live.append(t)


def test_truncating_into_a_shared_block_copies_it(model):
    pool = _pool(model)
    P = _prompt(100, 11)
    _publish(model, pool, P)
    b = model.session(pool=pool, max_ctx=256)
    assert b.attach_prefix(P) == 96
    b.truncate(40)                                   # inside shared block 1
    new = _prompt(30, 12)
    got = b.eval(new, all_rows=True)
    np.testing.assert_array_equal(got, _fresh(model, np.concatenate([P[:40], new]))[40:])
    # the published blocks are untouched: a later session still reproduces P
    c = model.session(pool=pool, max_ctx=256)
    assert c.attach_prefix(P) == 96
    np.testing.assert_array_equal(c.eval(P[96:], all_rows=True), _fresh(model, P)[96:])


def test_prefix_argument_errors(model):
    plain = model.pool(16)
    s = model.session(pool=plain, max_ctx=256)
    s.eval(_prompt(40, 13))
    with pytest.raises(ValueError):
        s.publish()                                  # the pool has no index
    pool = _pool(model, n_blocks=16)
    with pytest.raises(ValueError):
        pool.enable_prefix(4)                        # already enabled
    t = model.session(pool=pool, max_ctx=256)
    t.eval(_prompt(40, 14))
    with pytest.raises(ValueError):
        t.attach_prefix(_prompt(40, 14))             # not at position 0
    u = model.session(pool=pool, max_ctx=256)
    u.set_block_table([5, 6])
    with pytest.raises(ValueError):
        u.attach_prefix(_prompt(40, 15))             # a caller-fixed table
    with pytest.raises(ValueError):
        model.session(max_ctx=256).attach_prefix(_prompt(8, 16))   # contiguous session
