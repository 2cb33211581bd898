"""The pages' mutation gate run against the CUDA runtime ("Reproducing
Kipp", section "Mutation gate": planted addressing faults show that the
identity-layout tolerance gate and the adversarial block-table gate catch
different classes of defects).

A test build of the library (runtime.cu compiled with Q3_TEST_FAULTS, linked
into a separate library; the product never carries it) plants one fault in
what the host uploads, chosen by the Q3_FAULT environment variable.  Every
perturbed block id and slot stays inside the pool and inside the blocks the
session reserved, so no kernel reads or writes outside its buffers:
  1  read-block: the prefill attention reads through the identity table
     (entry i = block i), the writers through the real one;
  2  off-by-one slot: the K/V writer sees every row one position later;
  3  wrong block id: the prefill attention reads block id ^ 1;
  4  rollover: the writer puts block i's positions into the session's block
     i - 1.
Each runs in a child process (tests/fault_gate_child.py).  The expected
matrix (identity tolerance, adversarial table): no fault (pass, pass);
read-block (pass, FAIL) -- only the adversarial gate sees a layout the
readers ignore; off-by-one slot and rollover (FAIL, pass) -- the same defect
in every layout, which only the tolerance gate sees; wrong block id (FAIL,
FAIL).
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
EXPECTED = {0: (True, True), 1: (True, False), 2: (False, True), 3: (False, False), 4: (False, True)}


@pytest.fixture(scope="module")
def fault_lib():
    from qwen3_dense_decoder_gb300 import buildlib
    return buildlib.build_fault_variant()


@pytest.mark.parametrize("fault", sorted(EXPECTED))
def test_gates_catch_their_fault_classes(fault_lib, fault):
    env = dict(os.environ, Q3_FAULT=str(fault))
    r = subprocess.run([sys.executable, os.path.join(HERE, "fault_gate_child.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = json.loads(r.stdout.strip().splitlines()[-1])
    assert (got["identity_tolerance"], got["adversarial_table"]) == EXPECTED[fault], got
