"""The oracle under AddressSanitizer and UndefinedBehaviorSanitizer (the
pages' sanitizer gate: "Reproducing Kipp", section "Model-free gates", make
test-sanitize).  A sanitized copy of the oracle library is built in a
temporary directory and driven from a child process through every scheme,
both K/V storages, paged and contiguous sessions, batched rounds,
truncation and the prefix index under forced collisions and eviction; any
memory or undefined-behaviour error ends the child with a report."""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCENARIO = textwrap.dedent('''
    import sys
    sys.path.insert(0, sys.argv[1]); sys.path.insert(1, sys.argv[2])
    import numpy as np
    import oracle as orc
    assert orc.__file__.startswith(sys.argv[1]), orc.__file__
    from synthetic import AFFINE4, Q8_0, Shape, make_tokens, make_weights
    T = Shape("t", 2, 64, 4, 2, 32, 96, 128, True, rope_theta=1e4)
    for sh in (T, T.replace(scheme=Q8_0, tied=False), T.replace(scheme=AFFINE4), T.replace(kv_quant=Q8_0)):
        m = orc.Model(sh, make_weights(sh, seed=3), n_threads=3)
        toks = make_tokens(70, sh.vocab, seed=1)
        m.session(max_ctx=128).eval(toks, all_rows=True)
        pool = m.pool(12)
        pool.enable_prefix(0)
        a = m.session(pool=pool, max_ctx=128); a.eval(toks[:65]); a.publish()
        b = m.session(pool=pool, max_ctx=128); n = b.attach_prefix(toks); b.eval(toks[n:])
        b.truncate(40); b.eval(toks[:9])
        c = m.session(pool=pool, max_ctx=128); c.set_block_table([11, 10]); c.eval(toks[:50]); c.truncate(20)
        d = [m.session(pool=pool, max_ctx=128) for _ in range(3)]
        m.eval_batch(d, [toks[:5], toks[:33], toks[:12]])
        try:                                   # run the pool dry: evictions, then exhaustion
            for k in range(10):
                e = m.session(pool=pool, max_ctx=128); e.eval(make_tokens(40, sh.vocab, seed=50 + k)); d.append(e)
        except RuntimeError:
            pass
        del a, b, c, d
    w = np.random.default_rng(0).standard_normal((8, 256)).astype(np.float32) * 0.02
    orc.q8_0_unpack(orc.q8_0_pack(w), 256)
    orc.affine4_unpack(orc.affine4_pack(w), 256)
    print("scenario ok")
''')


def _runtime(name):
    gcc = shutil.which("gcc")
    if not gcc:
        return None
    path = subprocess.run([gcc, f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_oracle_is_clean_under_asan_and_ubsan(tmp_path):
    asan = _runtime("libasan.so")
    if not asan or not _runtime("libubsan.so"):
        pytest.skip("gcc's sanitizer runtimes are not installed")
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    for f in ("__init__.py", "q3_oracle.c", "q3_oracle.h"):
        shutil.copy(os.path.join(ROOT, "oracle", f), pkg / f)
    lib = pkg / "libq3_oracle.so"
    subprocess.check_call(["gcc", "-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
                           "-fno-omit-frame-pointer", "-std=c11", "-Wall", "-fPIC", "-shared", "-pthread",
                           "-o", str(lib), str(pkg / "q3_oracle.c"), "-lm"])
    os.utime(lib)                                      # newer than the sources: no rebuild
    env = dict(os.environ, LD_PRELOAD=asan, ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    script = tmp_path / "scenario.py"
    script.write_text(SCENARIO)
    r = subprocess.run([sys.executable, str(script), str(tmp_path), ROOT], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "scenario ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
