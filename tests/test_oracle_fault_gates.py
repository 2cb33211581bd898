"""The mutation gate ("Reproducing Kipp", section "Mutation gate"): faults
planted in the K/V read path show that the identity-layout tolerance gate
and the adversarial block-table gate catch different classes of addressing
defects.  The faults are the pages' four (1 read-block, 2 read-slot,
3 rollover, 4 K/V swap), written into the gather of a copy of the oracle
built in a temporary directory; the product code is never touched.

- tolerance gate: a paged session with the identity block table against the
  float64 brute force of tests/test_oracle_model.py (NMSE < 1e-6 per row,
  the pages' cached-vs-recompute bound; honest FP32-vs-FP64 differences stay
  below 3e-8 here);
- adversarial gate: paged sessions under seeded permuted tables against a
  contiguous session, bitwise.
A read that ignores the table hides behind the identity layout; a fault in
every layout's read path (K and V swapped) leaves paged and contiguous
equal; the others break both."""
import importlib.util
import os
import shutil
import subprocess

import numpy as np
import pytest

from synthetic import Shape, make_block_permutation, make_tokens, make_weights

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TINY = Shape("oracle-tiny", 2, 64, 4, 2, 16, 96, 128, True, rope_theta=1e4)
N_TOK = 100                                   # four blocks: past the rollover point

FAULT_READ = r'''
/* planted read-path fault (mutation gate) */
static uint8_t* fault_slot(orc_session* s, int l, int p, int is_v)
{
#if FAULT == 4
    is_v = !is_v;                                  /* K/V swap, every layout */
#endif
    if (!s->pool) return kv_slot(s, l, p, is_v);
    long blk = s->table[p / ORC_BLOCK], slot = p % ORC_BLOCK;
#if FAULT == 1
    blk = p / ORC_BLOCK;                           /* read-block: the table is ignored */
#elif FAULT == 2
    slot ^= 1;                                     /* read-slot */
#elif FAULT == 3
    blk = s->table[(p / ORC_BLOCK) % 2];           /* rollover after two blocks */
#endif
    uint8_t* base = is_v ? s->pool->v : s->pool->k;
    return base + (((long)l * s->pool->n_blocks + blk) * ORC_BLOCK + slot) * kv_row_bytes(&s->m->c);
}
'''

# fault -> (tolerance gate passes, adversarial gate passes)
EXPECTED = {0: (True, True), 1: (True, False), 2: (False, False), 3: (False, False), 4: (False, True)}


def _faulty_oracle(tmp_path, fault):
    pkg = tmp_path / f"fault{fault}" / "oracle"
    pkg.mkdir(parents=True)
    for f in ("__init__.py", "q3_oracle.h"):
        shutil.copy(os.path.join(ROOT, "oracle", f), pkg / f)
    src = open(os.path.join(ROOT, "oracle", "q3_oracle.c")).read()
    anchor = "/* ---- one round over a set of rows (one or more sessions) ---- */"
    reads = ("kv_load(c, kv_slot(s, j->layer, p, 0), K + p * kvr);",
             "kv_load(c, kv_slot(s, j->layer, p, 1), V + p * kvr);")
    assert src.count(anchor) == 1 and all(src.count(r) == 1 for r in reads)
    src = src.replace(anchor, FAULT_READ + "\n" + anchor)
    for r in reads:
        src = src.replace(r, r.replace("kv_slot(", "fault_slot("))
    (pkg / "q3_oracle.c").write_text(src)
    lib = pkg / "libq3_oracle.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-pthread", f"-DFAULT={fault}",
                           "-o", str(lib), str(pkg / "q3_oracle.c"), "-lm"])
    os.utime(lib)                                      # newer than the sources: no rebuild
    spec = importlib.util.spec_from_file_location(f"oracle_fault{fault}", pkg / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def tolerance_gate(orc, w, toks, ref) -> bool:
    m = orc.Model(TINY, w, n_threads=2)
    pool = m.pool(8)
    s = m.session(pool=pool, max_ctx=128)
    s.set_block_table(np.arange(4, dtype=np.int32))
    got = s.eval(toks, all_rows=True).astype(np.float64)
    return all(((got[t] - ref[t]) ** 2).sum() / (ref[t] ** 2).sum() < 1e-6 for t in range(len(toks)))


def adversarial_gate(orc, w, toks) -> bool:
    m = orc.Model(TINY, w, n_threads=2)
    ref = m.session(max_ctx=128).eval(toks, all_rows=True)
    for seed in (1, 2):
        pool = m.pool(16)
        s = m.session(pool=pool, max_ctx=128)
        s.set_block_table(make_block_permutation(16, seed)[:4])
        if not np.array_equal(s.eval(toks, all_rows=True), ref):
            return False
    return True


@pytest.fixture(scope="module")
def case():
    from test_oracle_model import brute_force_logits
    w = make_weights(TINY, seed=7)
    toks = make_tokens(N_TOK, TINY.vocab, seed=31)
    return w, toks, brute_force_logits(TINY, w, toks)


@pytest.mark.parametrize("fault", sorted(EXPECTED), ids=["none", "read-block", "read-slot", "rollover", "kv-swap"])
def test_gates_catch_the_planted_fault(tmp_path, case, fault):
    if not shutil.which("gcc"):
        pytest.skip("gcc is needed to build the planted-fault oracle")
    w, toks, ref = case
    orc = _faulty_oracle(tmp_path, fault)
    got = (tolerance_gate(orc, w, toks, ref), adversarial_gate(orc, w, toks))
    assert got == EXPECTED[fault], (fault, got)
