"""Child process of the GPU mutation gate (tests/test_gpu_fault_gates.py).

Loads the test build of the library (runtime.cu with Q3_TEST_FAULTS), plants
the fault named by Q3_FAULT, runs the two gates on the tiny shape and prints
one JSON line: {"fault": f, "identity_tolerance": bool, "adversarial_table": bool}.

- identity-layout tolerance gate: a session on the identity block table
  [0, 1, 2, 3] against the oracle, the usual comparison rule on the last row
  of each round;
- adversarial block-table gate: the same rounds on a permuted table that
  shares no block with the identity one, in a fresh pool, bitwise equal to
  the identity session's logits.

Rounds of 31, 32 and 37 tokens keep every perturbed write inside a reserved
block and never let two rows of one round write the same slot.
"""
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
import qwen3_dense_decoder_gb300 as q3  # noqa: E402
import synthetic  # noqa: E402
from helpers import check_row  # noqa: E402
from qwen3_dense_decoder_gb300 import buildlib  # noqa: E402

ROUNDS = (31, 32, 37)
PERMUTED = np.array([9, 14, 6, 11], np.int32)


def main():
    q3.LIB_PATH = buildlib.FAULT_LIB          # the test build, never the product library
    shape = synthetic.SHAPES["tiny"]
    w = synthetic.make_weights(shape, seed=901, device="cuda")
    model = q3.Model(shape, w, max_ctx=256, max_round_tokens=64)
    toks = synthetic.make_tokens(sum(ROUNDS), shape.vocab, seed=902)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")

    def run(table):
        pool = model.pool(16, 2)
        s = pool.session()
        s.set_block_table(table)
        out, a = [], 0
        for n in ROUNDS:
            s.eval(torch.tensor(toks[a:a + n], device="cuda"), logits)
            model.sync()
            out.append(logits.cpu().numpy().copy())
            a += n
        s.close()
        pool.close()
        return np.stack(out)

    ident = run(np.arange(4, dtype=np.int32))
    perm = run(PERMUTED)
    o = oracle.Model(shape, w).session(max_ctx=256)
    ref, a = [], 0
    for n in ROUNDS:
        ref.append(o.eval(toks[a:a + n]))
        a += n
    g1 = all(check_row(ident[i], ref[i]).ok for i in range(len(ROUNDS)))
    g2 = bool(np.array_equal(ident, perm))
    print(json.dumps({"fault": int(os.environ.get("Q3_FAULT", "0")), "identity_tolerance": g1,
                      "adversarial_table": g2}))


if __name__ == "__main__":
    main()
