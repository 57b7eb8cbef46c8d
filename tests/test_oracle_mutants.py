"""Plants plausible mistakes in copies of the oracle and checks that the pins
catch every one of them.

Each mutant is ``oracle.c`` with one textual change (a wrong index, a dropped
term, a shifted mask), compiled to a temporary library and run against the
pin tests in a child process (a mutant may also crash: that counts as caught).
The real oracle is never modified."""
import concurrent.futures
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = ["tests/test_oracle_attention.py", "tests/test_oracle_write.py",
        "tests/test_oracle_int8.py"]

# (name, text in oracle.c, replacement, occurrence to replace: 0-based or None for all)
MUTANTS = [
    ("kv-head-modulo", "int g = h / group;", "int g = h % hkv;", None),
    ("causal-ignores-ctx", "int64_t last = ctx + i;", "int64_t last = i;", None),
    ("ctx-off-by-one", "int64_t ctx = (int64_t)seq_lens[r] - n;",
     "int64_t ctx = (int64_t)seq_lens[r] - n - 1;", None),
    ("scale-dropped", "s *= scale;", "s *= 1.0;", None),
    ("max-not-subtracted", "scores[j] = exp(scores[j] - m);", "scores[j] = exp(scores[j]);", None),
    ("not-normalised", "double p = scores[j] / l;", "double p = scores[j];", None),
    ("key-block-index", "block_table[(int64_t)r * bt_row_stride + j / block_size]",
     "block_table[(int64_t)r * bt_row_stride + j % block_size]", 0),
    ("value-block-index", "block_table[(int64_t)r * bt_row_stride + j / block_size]",
     "block_table[(int64_t)r * bt_row_stride + (j + 1) / block_size]", 1),
    ("value-head-zero", "int64_t vrow = ((block * block_size + offset) * hkv + g) * d;",
     "int64_t vrow = ((block * block_size + offset) * hkv + 0) * d;", None),
    ("write-offset-zero", "int64_t offset = slot % block_size;", "int64_t offset = 0;", None),
    ("write-v-from-k", "value_cache[dst] = v[", "value_cache[dst] = k[", None),
    ("write-head-stride", "int64_t dst = ((block * block_size + offset) * hkv + h) * d + e;",
     "int64_t dst = ((block * block_size + offset) * hkv) * d + e;", None),
    ("query-row-ignores-request-start",
     "const uint16_t *qrow = q + (q0 + i) * q_row_stride + (int64_t)h * d;",
     "const uint16_t *qrow = q + i * q_row_stride + (int64_t)h * d;", None),
    ("query-head-uses-kv-head",
     "const uint16_t *qrow = q + (q0 + i) * q_row_stride + (int64_t)h * d;",
     "const uint16_t *qrow = q + (q0 + i) * q_row_stride + (int64_t)g * d;", None),
    ("key-head-zero", "int64_t krow = ((block * block_size + offset) * hkv + g) * d;",
     "int64_t krow = ((block * block_size + offset) * hkv + 0) * d;", None),
    ("key-offset-zero", "int64_t offset = j % block_size;", "int64_t offset = 0;", 0),
    ("key-excludes-itself", "for (int64_t j = 0; j <= last; ++j) {",
     "for (int64_t j = 0; j < last; ++j) {", 0),
    ("output-row-ignores-request-start",
     "double *orow = out + ((int64_t)query_start_loc[r] + i) * out_row_stride +",
     "double *orow = out + (i) * out_row_stride +", None),
    ("bt-width-check-strict", "if (nb > bt_width) return ORC_ERR_BT_WIDTH;",
     "if (nb >= bt_width) return ORC_ERR_BT_WIDTH;", None),
    ("block-id-check-dropped", "if (id < 0 || id >= num_blocks) return ORC_ERR_BLOCK_ID;", "",
     None),
    ("int8-truncates", "float r = rintf(x / scale);", "float r = truncf(x / scale);", None),
    ("int8-rounds-half-up", "float r = rintf(x / scale);", "float r = floorf(x / scale + 0.5f);",
     None),
    ("int8-no-clamp", "if (r > 127.0f) r = 127.0f;", "", None),
    ("int8-v-dequant-k-scale", "kv_value(value_cache, vrow + e, kv_int8, v_scale)",
     "kv_value(value_cache, vrow + e, kv_int8, k_scale)", None),
    ("int8-write-v-k-scale", "quantize_int8(v[t * v_row_stride + (int64_t)h * d + e], v_scale)",
     "quantize_int8(v[t * v_row_stride + (int64_t)h * d + e], k_scale)", None),
]


def _mutate(text, old, new, occurrence):
    assert old in text, old
    if occurrence is None:
        return text.replace(old, new)
    parts = text.split(old)
    assert len(parts) > occurrence + 1
    return old.join(parts[:occurrence + 1]) + new + old.join(parts[occurrence + 1:])


def _run_mutant(args):
    name, old, new, occ, tmp = args
    src = os.path.join(tmp, name + ".c")
    lib = os.path.join(tmp, name + ".so")
    with open(SRC) as f:
        text = f.read()
    with open(src, "w") as f:
        f.write(_mutate(text, old, new, occ))
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", lib,
                    "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=lib, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PINS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_planted_mistake_is_caught():
    with tempfile.TemporaryDirectory() as tmp:
        jobs = [(n, o, r, c, tmp) for n, o, r, c in MUTANTS]
        workers = max(1, min(len(jobs), os.cpu_count() or 1))
        with concurrent.futures.ThreadPoolExecutor(workers) as ex:
            results = dict(ex.map(_run_mutant, jobs))
    survivors = [n for n, rc in results.items() if rc == 0]
    assert not survivors, "pins missed planted mistakes: %s" % survivors


def test_unmutated_copy_passes_the_pins():
    """The harness itself: an unchanged copy must pass, or every mutant
    'caught' above would mean nothing."""
    with tempfile.TemporaryDirectory() as tmp:
        name, rc = _run_mutant(("identity", "int g = h / group;", "int g = h / group;", None, tmp))
    assert rc == 0
