"""Planted mistakes in the oracle must fail its pins (CPU only).

Each case copies oracle.c, plants one plausible mistake (a swapped index, a
dropped term, a wrong sign, a transposed operand, a wrong layout), builds the
copy into a temporary library and runs tests/test_oracle_pins.py against it in
a child process.  The pins are only worth something if every mistake fails at
least one of them.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = [
    ("block index and row swapped",
     "int32_t logical_block = p / B;\n        int32_t row = p % B;",
     "int32_t logical_block = p % B;\n        int32_t row = p / B;"),
    ("pool read as [N][B][Hkv][D]",
     "(((int64_t)phys * Hkv + g) * B + row) * D",
     "(((int64_t)phys * B + row) * Hkv + g) * D"),
    ("scale dropped", "x[i] = scale * dot;", "x[i] = dot;"),
    ("strided instead of contiguous head groups",
     "int32_t h = g * G + j;", "int32_t h = j * Hkv + g;"),
    ("exp sign flipped", "x[i] = exp(x[i] - m); den += x[i];", "x[i] = exp(m - x[i]); den += x[i];"),
    ("K and V swapped",
     "Kc[(int64_t)p * D + d] = load_as_double(k_pool", "Kc[(int64_t)p * D + d] = load_as_double(v_pool"),
    ("fp16 exponent off by one", "e - 25", "e - 24"),
    ("bf16 shifted wrongly", "(uint32_t)b << 16", "(uint32_t)b << 15"),
    ("normaliser dropped", "o[d] = acc / den;", "o[d] = acc;"),
    ("merge ignores the range maxima", "L += exp(m[k] - M) * l[k];", "L += l[k];"),
    ("partition ranges shifted", "int32_t first = k * P;", "int32_t first = k * P + 1;"),
    ("slot offset uses the block index",
     "(int64_t)phys * block_size + p % block_size", "(int64_t)phys * block_size + p / block_size"),
    ("write row from the wrong operator",
     "int64_t blk = slot / block_size, row = slot % block_size;",
     "int64_t blk = slot / block_size, row = slot / block_size;"),
    ("copy skips the V pool",
     "memcpy((char*)v_pool + (int64_t)dst", "if (0) memcpy((char*)v_pool + (int64_t)dst"),
    ("swap copies K into V",
     "memcpy((char*)dst_v + (int64_t)dst * block_bytes, (const char*)src_v",
     "memcpy((char*)dst_v + (int64_t)dst * block_bytes, (const char*)src_k"),
    ("multi-query sees one position too many",
     "int32_t c = ctx - nq + 1 + j;", "int32_t c = ctx - nq + 2 + j;"),
    ("copy-on-write skipped for shared blocks",
     "            if (refcount[b] > 1) {\n                int32_t nb = take_free",
     "            if (refcount[b] > 99) {\n                int32_t nb = take_free"),
    ("freed blocks never return to the stack",
     "if (refcount[b] == 0) free_ids[(*free_count)++] = b;", "(void)0;"),
    ("merge normaliser dropped", "            o[d] = acc / L;", "            o[d] = acc;"),
    ("merge skips the first range",
     "for (int32_t k = 0; k < max_parts; ++k) if (l[k] > 0.0) L += exp(m[k] - M) * l[k];",
     "for (int32_t k = 1; k < max_parts; ++k) if (l[k] > 0.0) L += exp(m[k] - M) * l[k];"),
    ("padding position mapped to a slot",
     "if (p < 0) { slot_mapping[t] = -1; continue; }",
     "if (p < -1) { slot_mapping[t] = -1; continue; }"),
    ("fork adds no reference", "            refcount[b] += 1;", "            refcount[b] += 0;"),
    ("free leaves the table row", "            row[j] = -1;\n", "            (void)0;\n"),
    ("slot mapping ignores the token's sequence",
     "int32_t s = token_seq ? token_seq[t] : t;", "int32_t s = t;"),
    ("partition drops its last position",
     "int32_t n = ctx - first < P ? ctx - first : P;",
     "int32_t n = ctx - first < P ? ctx - first - 1 : P - 1;"),
    ("partition range maximum not subtracted",
     "for (int32_t i = 0; i < n; ++i) { x[i] = exp(x[i] - m); l += x[i]; }",
     "for (int32_t i = 0; i < n; ++i) { x[i] = exp(x[i]); l += x[i]; }"),
    ("block copy direction reversed",
     "memcpy((char*)k_pool + (int64_t)dst * block_bytes, (const char*)k_pool + (int64_t)src * block_bytes,",
     "memcpy((char*)k_pool + (int64_t)src * block_bytes, (const char*)k_pool + (int64_t)dst * block_bytes,"),
    ("q rows read head-major",
     "qd[d] = load_as_double(q, dtype, ((int64_t)s * Hq + h) * D + d);\n            if (ctx == 0)",
     "qd[d] = load_as_double(q, dtype, ((int64_t)h * num_seqs + s) * D + d);\n            if (ctx == 0)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    with open(SRC) as f:
        text = f.read()
    assert old in text, "mutation site not found: " + name
    bad = tmp_path / "oracle_mutant.c"
    bad.write_text(text.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fopenmp", str(bad), "-o", str(so), "-lm"], check=True,
                   capture_output=True)
    env = dict(os.environ, ORACLE_LIB=str(so))
    proc = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, "no pin caught the planted mistake: " + name
