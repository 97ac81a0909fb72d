"""The oracle's pins catch plausible mistakes in the oracle.

Each case plants one mistake (a dropped term, a wrong sign, index or bound,
a swapped operand) in a copy of ``oracle/`` made in a scratch directory of
the repository (``.oracle_mutants/``, ignored by git, removed afterwards),
then runs the pin suites (tests/test_oracle.py, tests/test_oracle_fp8.py)
against that copy in a child process: at least one pin must fail.  A control
run of the unchanged copy must pass, so a surviving mistake cannot hide
behind a broken harness.  The repository's own oracle is never modified, and
nothing here touches a GPU.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = [os.path.join(ROOT, "tests", "test_oracle.py"),
        os.path.join(ROOT, "tests", "test_oracle_fp8.py")]

C, PY, FP8 = "attention.c", "__init__.py", "fp8.py"

# (name, file, text, replacement): the text must occur exactly once
MUTANTS = [
    # addressing: P2 "Page-table 寻址" / P1 §3
    ("slot drops the offset", C,
     "*slot = phys * block_size + offset;", "*slot = phys * block_size;"),
    ("slot ignores the table", C,
     "int64_t phys = table[logical];", "int64_t phys = logical;"),
    ("slot offset from the logical index", PY,
     "return phys * block_size + offset", "return phys * block_size + logical"),
    ("negative physical id accepted", PY,
     "    if phys < 0:\n        raise ValueError", "    if phys < -1:\n        raise ValueError"),
    # attention arithmetic (one output row)
    ("score without the scale", C,
     "        x[i] = scale * dot;\n    }\n    double m = x[0];",
     "        x[i] = dot;\n    }\n    double m = x[0];"),
    ("max added instead of subtracted", C,
     "        double w = exp(x[i] - m);\n        denom += w;\n        int64_t slot;\n"
     "        orc_physical_slot(table, n_entries",
     "        double w = exp(m - x[i]);\n        denom += w;\n        int64_t slot;\n"
     "        orc_physical_slot(table, n_entries"),
    ("no division by the softmax sum", C,
     "    for (int32_t d = 0; d < D; ++d) out[d] /= denom;\n", ""),
    ("V read from the K pool", C,
     "out[d] += w * elem(vpool, dtype, vrow + d);", "out[d] += w * elem(kpool, dtype, vrow + d);"),
    ("K rows of kv-head 0 only", C,
     "if (blk >= num_blocks) return -2;\n        size_t krow = (((size_t)blk * Hkv + h) * Bp",
     "if (blk >= num_blocks) return -2;\n        size_t krow = (((size_t)blk * Hkv + 0) * Bp"),
    ("bf16 bits misplaced", C,
     "uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;",
     "uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 15;"),
    ("first key left out of the max", C,
     "    double m = x[0];\n    for (int64_t i = 1; i < n_vis; ++i) if (x[i] > m) m = x[i];",
     "    double m = x[n_vis - 1];\n    for (int64_t i = 1; i < n_vis - 1; ++i) if (x[i] > m) m = x[i];"),
    # GQA mapping and the visible length of decode
    ("GQA heads interleaved instead of grouped", C,
     "max_blocks, g / G, context_lens[s], scale", "max_blocks, g % Hkv, context_lens[s], scale"),
    ("decode skips the newest token", C,
     "max_blocks, g / G, context_lens[s], scale", "max_blocks, g / G, context_lens[s] - 1, scale"),
    # split-KV merge (P1 §4 state combination)
    ("merge drops the sum rescale", C, "L += pl[p] * c;", "L += pl[p];"),
    ("merge drops the value rescale", C,
     "o[d] += pa[p * D + d] * c;", "o[d] += pa[p * D + d];"),
    ("partition max from the last partition only", C,
     "for (int64_t p = 1; p < nparts; ++p) if (pm[p] > M) M = pm[p];",
     "M = pm[nparts - 1];"),
    # prefill
    ("new tokens placed at the start of the context", C,
     "int64_t pos = context_lens[s] - n_new + i;", "int64_t pos = i;"),
    ("causal row sees one token more", C,
     "int64_t n_vis = causal ? pos + 1 : context_lens[s];",
     "int64_t n_vis = causal ? (pos + 2 < context_lens[s] ? pos + 2 : context_lens[s]) "
     ": context_lens[s];"),
    ("non-causal row sees only the past", C,
     "int64_t n_vis = causal ? pos + 1 : context_lens[s];", "int64_t n_vis = pos + 1;"),
    # sliding window
    ("window one token short", C,
     "int64_t lo = (window > 0 && n > window) ? n - window : 0;",
     "int64_t lo = (window > 0 && n > window) ? n - window + 1 : 0;"),
    ("window one token long", C,
     "int64_t lo = (window > 0 && n > window) ? n - window : 0;",
     "int64_t lo = (window > 0 && n > window) ? n - window - 1 : 0;"),
    # contiguous layout of P4 (paged == contiguous pin)
    ("contiguous K of kv-head 0 only", C,
     "size_t krow = (((size_t)s * max_seq + i) * Hkv + h) * D;",
     "size_t krow = (((size_t)s * max_seq + i) * Hkv + 0) * D;"),
    # ownership: P2 "引用计数与尾块 COW" / "生命周期与所有权"
    ("fork does not count the new holder", PY,
     "        for b in child:\n            self.refcount[b] += 1\n",
     "        for b in child:\n            pass\n"),
    ("shared tail written in place", PY,
     "if self.refcount[cur] > 1:", "if self.refcount[cur] > 2:"),
    ("copy-on-write keeps the old holder", PY,
     "                self.refcount[cur] -= 1\n", ""),
    ("released block never freed", PY,
     "            if self.refcount[b] == 0:\n                self.free.append(b)\n", ""),
    ("new block appended mid-table", PY,
     "            if logical != len(table):\n                raise ValueError",
     "            if logical > len(table):\n                raise ValueError"),
    # pool writes and copies (P1 §4.1, P1 §5)
    ("V row written with K", PY,
     "        vpool[blk, :, off, :] = v_new[t]", "        vpool[blk, :, off, :] = k_new[t]"),
    ("block copy runs backwards", PY,
     "        kpool[b] = kpool[a]", "        kpool[a] = kpool[b]"),
    ("negative slot accepted", PY,
     "        if slot < 0 or slot >= N * Bp:", "        if slot < -1 or slot >= N * Bp:"),
    # E4M3 format and row scales (OCP 8-bit floating point)
    ("mantissa weight halved", FP8, "(1.0 + m / 8.0)", "(1.0 + m / 16.0)"),
    ("subnormal step 2^-10", FP8, "m / 8.0 * 2.0 ** -6", "m / 8.0 * 2.0 ** -7"),
    ("ties to the odd code", FP8, "((hi & 1) == 0)", "((hi & 1) == 1)"),
    ("ties away from zero", FP8, "((d_hi == d_lo) & ((hi & 1) == 0))", "(d_hi == d_lo)"),
    ("sign bit dropped", FP8,
     "    code = code | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)\n", ""),
    ("scale from 240 instead of 448", FP8,
     "scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)",
     "scale = (amax / np.float32(240.0)).astype(np.float32)"),
    ("dequantise divides by the scale", FP8,
     "return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]",
     "return e4m3_decode(codes) / np.asarray(scales, dtype=np.float64)[..., None]"),
]


def _copy_oracle(dst_root, mutant=None):
    dst = os.path.join(dst_root, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst,
                    ignore=shutil.ignore_patterns("*.so", "*.so.*", "__pycache__"))
    if mutant is not None:
        _, fname, old, new = mutant
        path = os.path.join(dst, fname)
        with open(path, encoding="utf-8") as f:
            src = f.read()
        assert src.count(old) == 1, "mutation site not unique in %s: %r" % (fname, old[:60])
        with open(path, "w", encoding="utf-8") as f:
            f.write(src.replace(old, new))
    return dst_root


SCRATCH = os.path.join(ROOT, ".oracle_mutants")


def _run_pins(work):
    tmp = os.path.join(work, "tmp")
    os.makedirs(tmp, exist_ok=True)
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([work, ROOT]), OMP_NUM_THREADS="2",
               PYTHONDONTWRITEBYTECODE="1", TMPDIR=tmp)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PINS], cwd=work, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-1500:] + r.stderr[-1500:]


@pytest.fixture
def scratch():
    shutil.rmtree(SCRATCH, ignore_errors=True)
    os.makedirs(SCRATCH)
    yield SCRATCH
    shutil.rmtree(SCRATCH, ignore_errors=True)


def test_every_planted_mistake_fails_a_pin(scratch):
    control = _copy_oracle(os.path.join(scratch, "control"))
    rc, log = _run_pins(control)
    assert rc == 0, "the unchanged copy of the oracle must pass its pins:\n" + log

    def one(i):
        work = _copy_oracle(os.path.join(scratch, "m%02d" % i), MUTANTS[i])
        return i, _run_pins(work)

    survivors, crashed = [], []
    with cf.ThreadPoolExecutor(max_workers=6) as pool:
        for i, (rc, log) in pool.map(one, range(len(MUTANTS))):
            if rc == 0:
                survivors.append(MUTANTS[i][0])
            elif rc != 1:  # 1 = tests failed; anything else is a crash or a usage error
                crashed.append("%s (rc %d): %s" % (MUTANTS[i][0], rc, log[-400:]))
    assert not crashed, "mutants that did not run to a failing pin:\n" + "\n".join(crashed)
    assert not survivors, "planted mistakes no pin caught: " + ", ".join(survivors)


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutation_sites_exist(mutant):
    # every mutation site is still present once, so an edit of the oracle
    # cannot quietly turn a case into a no-op
    _, fname, old, _ = mutant
    with open(os.path.join(ROOT, "oracle", fname), encoding="utf-8") as f:
        assert f.read().count(old) == 1
