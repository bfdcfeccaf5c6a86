"""Each plausible mistake planted in a copy of the oracle (its C source, or
its Python allocator rules) must make the oracle's pin suite
(tests/test_oracle.py) fail -- evidence that the pins pin the arithmetic and
the rules, not just exercise them.  CPU only: C mutants are compiled with
gcc into a temporary directory, Python mutants run from a temporary copy of
the tree; the committed oracle is untouched."""
import os
import shutil
import subprocess
import sys

import pytest

from tests.conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "pagedkv_oracle.c")

# (name, exact source text, planted replacement) -- every occurrence is replaced
MUTANTS = [
    ("gqa head mapping", "int kvh = h / group;", "int kvh = h % n_kv_heads;"),
    ("row inside the block", "size_t row = (size_t)(t % block_size);",
     "size_t row = (size_t)((t + 1) % block_size);"),
    ("block of a token", "[(size_t)s * max_blocks_per_seq + t / block_size];",
     "[(size_t)s * max_blocks_per_seq + (t + 1) / block_size];"),
    ("scale dropped", "x[t] = scale * acc;", "x[t] = acc;"),
    ("K and V swapped in the scores", "double ki = orc_load(k_pool,", "double ki = orc_load(v_pool,"),
    ("no normalisation", "double w = exp(x[t] - m) / z;", "double w = exp(x[t] - m);"),
    ("maximum pass inverted", "if (x[t] > m)", "if (x[t] < m)"),
    ("sum pass off by one", "for (int t = 0; t < n; ++t)\n                z += exp(x[t] - m);",
     "for (int t = 1; t < n; ++t)\n                z += exp(x[t] - m);"),
    ("online carry not rescaled", "double carry = L * exp(M - M_new);", "double carry = L;"),
    ("online weights not divided", "o[i] = (carry / L_new) * o[i] + acc_v[i] / L_new;",
     "o[i] = (carry / L_new) * o[i] + acc_v[i];"),
    ("merge weight of the new part", "double part = l[k] * exp(m[k] - M_new);",
     "double part = l[k];"),
    ("copy direction reversed",
     "memmove((char*)dst_pool + j * block_bytes, (const char*)src_pool + i * block_bytes,",
     "memmove((char*)dst_pool + i * block_bytes, (const char*)src_pool + j * block_bytes,"),
    ("append row", "int64_t row = slot % block_size;", "int64_t row = (slot + 1) % block_size;"),
    ("fp16 exponent bias", "mag = ldexp((double)(1024 + frac), expo - 25);",
     "mag = ldexp((double)(1024 + frac), expo - 24);"),
    ("bf16 subnormals dropped", "mag = ldexp((double)frac, -133);", "mag = 0.0;"),
    ("kv bytes without the K/V factor", "return 2u * elem_bytes * n_layers",
     "return elem_bytes * n_layers"),
    ("query rows reversed", "int row = q_start[s] + i;", "int row = q_start[s] + (q_len - 1 - i);"),
    ("causal window one short", "int cnt = pos + 1;", "int cnt = pos > 0 ? pos : 1;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation site for '{name}' not found: update the mutant list"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(mutant), "-lm"], check=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(so))
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True)
    assert res.returncode != 0, f"the pins did not catch: {name}\n{res.stdout[-2000:]}"


BM_SRC = os.path.join(ROOT, "oracle", "block_manager.py")

# (name, exact source text, planted replacement) in oracle/block_manager.py
PY_MUTANTS = [
    ("highest free id first", "    for b, r in enumerate(refs):\n        if r == 0:\n            refs[b] = 1",
     "    for b, r in reversed(list(enumerate(refs))):\n        if r == 0:\n            refs[b] = 1"),
    ("page opened at n mod B == 1", "    if num_tokens % block_size == 0:\n        b = take_block(refs)",
     "    if num_tokens % block_size == 1:\n        b = take_block(refs)"),
    ("dropped reference never freed", "        refs[b] -= 1", "        refs[b] -= 0"),
    ("token row shifted", "    return table[n // block_size] * block_size + n % block_size",
     "    return table[n // block_size] * block_size + (n + 1) % block_size"),
]


def _copy_tree(dst):
    ignore = shutil.ignore_patterns("_build", "__pycache__", "*.so", "*.o", "csrc")
    for d in ("oracle", "tests", "paged_kv_decode_26_gb300"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d), ignore=ignore)
    shutil.copy(os.path.join(ROOT, "pytest.ini"), dst)


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_pins_catch_planted_allocator_mistake(tmp_path, name, old, new):
    from oracle import build as ob
    src = open(BM_SRC).read()
    assert src.count(old) == 1, f"mutation site for '{name}' not found: update the mutant list"
    _copy_tree(str(tmp_path))
    with open(os.path.join(str(tmp_path), "oracle", "block_manager.py"), "w") as f:
        f.write(src.replace(old, new))
    env = dict(os.environ, PKV_ORACLE_LIB=ob.build())
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                          os.path.join("tests", "test_oracle.py")],
                         cwd=str(tmp_path), env=env, capture_output=True, text=True)
    assert res.returncode != 0, f"the pins did not catch: {name}\n{res.stdout[-2000:]}"
    assert "passed" in res.stdout or "failed" in res.stdout, res.stdout[-2000:]


def test_unmutated_copy_passes(tmp_path):
    """The copied tree itself passes the pins (so a mutant's failure is the
    mutant's)."""
    from oracle import build as ob
    _copy_tree(str(tmp_path))
    env = dict(os.environ, PKV_ORACLE_LIB=ob.build())
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                          os.path.join("tests", "test_oracle.py")],
                         cwd=str(tmp_path), env=env, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout[-3000:]
