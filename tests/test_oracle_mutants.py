"""Each plausible mistake planted in a copy of the oracle's C source must make
the oracle's pin suite (tests/test_oracle.py) fail -- evidence that the pins
pin the arithmetic, not just exercise it.  CPU only: the mutants are compiled
with gcc into a temporary directory; the committed oracle is untouched."""
import os
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
