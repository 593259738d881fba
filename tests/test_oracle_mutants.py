"""The pins have teeth: plant a plausible mistake in a copy of the oracle's C
source (on the CPU), rebuild it, and check that at least one pin fails.

Each mutant runs in a child process, so a mutant that crashes counts as caught
and cannot take the test run down with it."""
import json
import os
import subprocess
import sys

import pytest

import oracle

MUTANTS = [
    ("causal window one short", "int64_t n_keys = p + 1;", "int64_t n_keys = p;"),
    ("top-left causal alignment", "int64_t p = Lk - Lq + i;", "int64_t p = i;"),
    ("GQA map h % Hkv", "int64_t hk = h / group;", "int64_t hk = h % Hkv;"),
    ("scale dropped", "s[t] = scale * dot;", "s[t] = dot;"),
    ("scale squared", "s[t] = scale * dot;", "s[t] = scale * scale * dot;"),
    ("max subtracted with the wrong sign", "double w = exp(s[t] - m);", "double w = exp(m - s[t]);"),
    ("normalisation dropped", "out[j] = out[j] / denom;", "out[j] = out[j] / (double)n_keys;"),
    ("value operand read from keys",
     "out[j] += w * elem_to_double(vrows[t][j], elem);", "out[j] += w * elem_to_double(krows[t][j], elem);"),
    ("in-block offset transposed", "int64_t slot = block * block_size + t % block_size;",
     "int64_t slot = block * block_size + t / block_size;"),
    ("head offset dropped in gather", "krows[t] = k_cache + slot * D + hk * head_dim;",
     "krows[t] = k_cache + slot * D;"),
    ("store ignores the row stride", "k_cache[slot * D + e] = k[i * k_row_stride + e];",
     "k_cache[slot * D + e] = k[i * D + e];"),
    ("decode context excludes the new token", "int64_t n_keys = context_lens[b];",
     "int64_t n_keys = context_lens[b] - 1;"),
    ("query read from the wrong head", "qd[j] = elem_to_double(q[token * q_row_stride + h * head_dim + j], elem);",
     "qd[j] = elem_to_double(q[token * q_row_stride + hk * head_dim + j], elem);"),
    ("fp16 exponent bias off by one", "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)(1024 + f), e - 24);"),
    ("fp16 implicit leading one dropped", "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)f, e - 15);"),
    ("fp16 subnormal scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -14);"),
    ("fp16 read as bf16", "return elem == ORACLE_ELEM_F16 ? f16_to_double(bits) : bf16_to_double(bits);",
     "return bf16_to_double(bits);"),
]

_CHILD = r"""
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
orc = oracle.Oracle({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(orc)
    except Exception as e:
        failed.append(pin.__name__)
print(json.dumps(failed))
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {old}"
    mutated = src.replace(old, new)
    assert mutated != src
    csrc = tmp_path / "mutant.c"
    csrc.write_text(mutated)
    lib = str(tmp_path / "libmutant.so")
    oracle.build(str(csrc), lib, force=True)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = _CHILD.format(root=root, tests=os.path.dirname(os.path.abspath(__file__)), lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    if r.returncode != 0:
        return          # the mutant crashed the child: caught
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed, f"no pin caught mutant '{name}'"
