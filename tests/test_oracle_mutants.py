"""Planted mistakes: do the oracle's pins catch them?

Each mutant below is a copy of oracle/mc2_oracle.c with one plausible mistake
written into it: a dropped term, a wrong sign, index or exponent bias, a
transposed operand, another rounding rule, the steps in another order.  The
copy is compiled on its own, and the oracle's pin tests
(tests/test_oracle_*.py, which check the oracle against closed forms, brute
force, hand-worked values and independent library routines) are run against
it in a child process through MC2_ORACLE_LIB.  Every mutant must make at least
one pin fail; the unchanged copy, built the same way, must pass them all.

The same is done for the oracle's Python wrapper (oracle/__init__.py: the
argument conversions and the exact fp64 route of large int8 products): a copy
of the package with one mistake is imported first in the child process, so it
stands in for the committed one.

The mistakes are planted on the CPU only, in copies under pytest's temporary
folder; the committed oracle is never modified.  A mutant whose mistake cannot
change any result (an equivalent mutant) does not belong in these lists, nor
one that would make the C code write past a buffer.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mc2_oracle.c")
PY_SRC = os.path.join(ROOT, "oracle", "__init__.py")
PINS = sorted(os.path.join(ROOT, "tests", f) for f in os.listdir(os.path.join(ROOT, "tests"))
              if f.startswith("test_oracle_") and f.endswith(".py") and f != "test_oracle_mutants.py")

# name -> (text in mc2_oracle.c, replacement); the text must occur exactly once
MUTANTS = {
    # 16-bit conversions (IEEE binary16 / bfloat16 layouts)
    "decode16 subnormal exponent off by one": (
        "r = ldexp((double)f, 1 - bias - fb);", "r = ldexp((double)f, -bias - fb);"),
    "encode16 rounds ties away from zero": (
        "double r = nearbyint(s);", "double r = round(s);"),
    "encode16 drops the carry into the next binade": (
        "if (ri == (1u << (fb + 1))) {", "if (0) {"),
    "encode16 treats subnormals as normals": (
        "if (E < emin) E = emin;", "(void)emin;"),
    "decode16 reads NaN patterns as infinity": (
        "r = f ? NAN : INFINITY;", "r = INFINITY;"),
    "encode16 turns NaN into infinity": (
        "if (isnan(x)) return (uint16_t)(sign | inf | (1u << (fb - 1)));",
        "if (isnan(x)) return (uint16_t)(sign | inf);"),
    "encode16 loses the sign of zero": (
        "if (a == 0.0) return sign;", "if (a == 0.0) return 0;"),
    "encode16 wraps on overflow": (
        "if (efield >= (1u << eb) - 1u) return (uint16_t)(sign | inf);", "(void)inf;"),
    # AllGatherMatmul
    "AG interleaves the shards instead of concatenating them": (
        "int64_t r = i / m_local;          /* which rank's shard */\n"
        "                int64_t li = i - r * m_local;     /* row inside that shard */",
        "int64_t r = i % world_size;\n                int64_t li = i / world_size;"),
    "AG reads the (n, k) weight as (k, n)": (
        "s += (double)tab[arow[kk]] * (double)tab[wrow[kk]];",
        "s += (double)tab[arow[kk]] * (double)tab[x2[kk * n + j]];"),
    "AG drops the last k term": (
        "for (int64_t kk = 0; kk < k; ++kk) {\n                        double a = tab[arow[kk]];",
        "for (int64_t kk = 0; kk < k - 1; ++kk) {\n                        double a = tab[arow[kk]];"),
    "gather stacks the shards in reverse rank order": (
        "memcpy(gathered + (int64_t)r * m_local * k, chunks[r],",
        "memcpy(gathered + (int64_t)r * m_local * k, chunks[world_size - 1 - r],"),
    "AG ignores the requested rows": (
        "int64_t i = rows ? rows[ii] : ii;\n                int64_t r = i / m_local;",
        "int64_t i = ii;\n                int64_t r = i / m_local;"),
    "AG drops the bias": (
        "double v = acc[j] + (bias ? (double)tab[bias[j]] : 0.0);", "double v = acc[j];"),
    "AG rounds before adding the bias": (
        "double v = acc[j] + (bias ? (double)tab[bias[j]] : 0.0);",
        "double v = (double)tab[oracle_encode16_rne(acc[j], is_bf16)] + (bias ? (double)tab[bias[j]] : 0.0);"),
    # AlltoAllQuantMatmul: permute, commOut, quant, int8 product, dequant
    "permute interleaves the ranks' elements": (
        "int64_t dst = ii * cols + (int64_t)r * h + hh;", "int64_t dst = ii * cols + hh * rank_size + r;"),
    "commOut stacks (token, rank) instead of (rank, token)": (
        "int64_t dst = ((int64_t)r * bs_local + t) * h + hh;",
        "int64_t dst = ((int64_t)t * rank_size + r) * h + hh;"),
    "permute ignores the requested rows": (
        "int64_t t = rows ? rows[ii] : ii;\n        if (t < 0 || t >= bs_local) return OR_ERR_ARG;\n        for (int r",
        "int64_t t = ii;\n        if (t < 0 || t >= bs_local) return OR_ERR_ARG;\n        for (int r"),
    "quant takes the signed maximum instead of the absolute one": (
        "float ay = fabsf(y);", "float ay = y;"),
    "int8 product reads the activations as unsigned": (
        "int64_t av = a[t * k + kk];", "int64_t av = (uint8_t)a[t * k + kk];"),
    "dequant takes the x1 scale by column": (
        "v = v * x1_scale[t];\n            v = v * x2_scale[j];",
        "v = v * x1_scale[j % n_rows];\n            v = v * x2_scale[j];"),
    "quant divides the absmax by 128": (
        "float scale = amax / 127.0f;", "float scale = amax / 128.0f;"),
    "quant truncates": (
        "float rv = nearbyintf(v);", "float rv = truncf(v);"),
    "quant rounds ties away from zero": (
        "float rv = nearbyintf(v);", "float rv = roundf(v);"),
    "quant multiplies by the reciprocal of the scale": (
        "float v = y / scale;", "float v = y * (1.0f / scale);"),
    "quant leaves the smooth scale out of the absmax": (
        "float s = smooth ? (float)oracle_decode16(smooth[c], is_bf16) : 1.0f;\n"
        "            float y = x * s;\n            float ay",
        "float s = 1.0f;\n            float y = x * s;\n            float ay"),
    "int8 product reads x2 as unsigned": (
        "s[j] += av * (int64_t)brow[j];", "s[j] += av * (int64_t)(uint8_t)brow[j];"),
    "int8 product misses an int32 overflow": (
        "if (s[j] > INT32_MAX || s[j] < INT32_MIN) {", "if (0) {"),
    "dequant drops the x2 scale": (
        "v = v * x2_scale[j];", "(void)x2_scale;"),
    "dequant drops the bias": (
        "if (bias) v = v + bias[j];", "(void)bias;"),
    "dequant applies the scales in the other order": (
        "v = v * x1_scale[t];\n            v = v * x2_scale[j];",
        "v = v * x2_scale[j];\n            v = v * x1_scale[t];"),
    "dequant rounds to fp16": (
        "out_bf16[t * n + j] = oracle_encode16_rne((double)v, 1);",
        "out_bf16[t * n + j] = oracle_encode16_rne((double)v, 0);"),
    "full quant takes the scale of the output row, not of the token": (
        "sc[ii] = ((const float *)x1_scale_in)[t];", "sc[ii] = ((const float *)x1_scale_in)[ii];"),
    # MatmulReduceScatter
    "reduce-scatter leaves rank 0 out of the sum": (
        "for (int r = 0; r < world_size; ++r) {        /* the reduction over ranks */",
        "for (int r = 1; r < world_size; ++r) {"),
    "reduce-scatter reads the (n, k) weight as (k, n)": (
        "uint16_t wv = w_is_nk ? w_chunks[r][j * k_local + kk] : w_chunks[r][kk * n + j];",
        "uint16_t wv = w_chunks[r][kk * n + j];"),
    "reduce-scatter ignores the requested rows": (
        "int64_t i = rows ? rows[ii] : ii;\n        for (int64_t j = 0; j < n; ++j) {\n            double s = 0.0;",
        "int64_t i = ii;\n        for (int64_t j = 0; j < n; ++j) {\n            double s = 0.0;"),
    "reduce-scatter drops the bias": (
        "if (bias) s += (double)tab[bias[j]];\n            out[ii * n + j] = oracle_encode16_rne(s, is_bf16);",
        "out[ii * n + j] = oracle_encode16_rne(s, is_bf16);"),
    # weight and bias gradients
    "weight gradient reads dY untransposed": (
        "double a = (double)tab[dy[t * n + i]];", "double a = (double)tab[dy[i * m + t]];"),
    "weight gradient reverses the columns of X": (
        "acc[j] += a * (double)tab[xrow[j]];", "acc[j] += a * (double)tab[xrow[k - 1 - j]];"),
    "weight gradient ignores the requested rows": (
        "int64_t i = rows ? rows[ii] : ii;\n            for (int64_t j = 0; j < k; ++j) acc[j] = 0.0;",
        "int64_t i = ii;\n            for (int64_t j = 0; j < k; ++j) acc[j] = 0.0;"),
    "bias gradient leaves out the first row": (
        "for (int64_t t = 0; t < m; ++t) s += (double)tab[dy[t * n + i]];",
        "for (int64_t t = 1; t < m; ++t) s += (double)tab[dy[t * n + i]];"),
    # QuantAllReduce and its element formats
    "e4m3 exponent bias 8": (
        "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3 takes its NaN code for a number": (
        "if (e == 15 && m == 7) return NAN;", "(void)0;"),
    "e5m2 subnormal scale 2^-15": (
        "ldexp((double)m / 4.0, -14)", "ldexp((double)m / 4.0, -15)"),
    "e5m2 reads its infinities as NaN": (
        "if (e == 31) return m == 0 ? (sign ? -INFINITY : INFINITY) : NAN;", "if (e == 31) return NAN;"),
    "e8m0 bias 128": (
        "return ldexp(1.0, (int)v - 127);", "return ldexp(1.0, (int)v - 128);"),
    "all-reduce picks the fp32 scale of the wrong group": (
        "(double)((const float *)scale_chunks[r])[t * groups + j / G]",
        "(double)((const float *)scale_chunks[r])[t * groups + j % groups]"),
    "all-reduce picks the e8m0 scale of the wrong group": (
        ": oracle_decode_e8m0(((const uint8_t *)scale_chunks[r])[t * groups + j / G]);",
        ": oracle_decode_e8m0(((const uint8_t *)scale_chunks[r])[t * groups + j % groups]);"),
    "all-reduce leaves out the last rank": (
        "for (int r = 0; r < world_size; ++r) {\n                uint8_t xv",
        "for (int r = 0; r < world_size - 1; ++r) {\n                uint8_t xv"),
    "all-reduce reads int8 codes as unsigned": (
        "double x = x_kind == 0 ? (double)(int8_t)xv :", "double x = x_kind == 0 ? (double)xv :"),
}


# name -> [(text in oracle/__init__.py, replacement), ...]; each text occurs exactly once
PY_MUTANTS = {
    "the fp64 route of the int8 product sums in fp32": [
        ("    ad = ac.double()\n", "    ad = ac.float()\n"),
        ("blk = ad @ bc[:, j0:j0 + col_block].double()", "blk = ad @ bc[:, j0:j0 + col_block].float()")],
    "the fp64 route takes every token's scale for a row subset": [
        ("sc = s_in if r is None else s_in[r]", "sc = s_in")],
    "bf16 tensors passed as fp16": [
        ("    if dtype == torch.bfloat16:\n        return 1", "    if dtype == torch.bfloat16:\n        return 0")],
    "e4m3 and e5m2 codes swapped": [
        ('X_KINDS = {"int8": 0, "e4m3": 1, "e5m2": 2}', 'X_KINDS = {"int8": 0, "e4m3": 2, "e5m2": 1}')],
    "fp32 and e8m0 scales swapped": [
        ('SCALE_KINDS = {"fp32": 0, "e8m0": 1}', 'SCALE_KINDS = {"fp32": 1, "e8m0": 0}')],
    "fp16 and bf16 outputs swapped": [
        ("_OUT_KINDS = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}",
         "_OUT_KINDS = {torch.float32: 0, torch.float16: 2, torch.bfloat16: 1}")],
    "AG bias converted to fp16 whatever the operands": [
        ("b = None if bias is None else _c(bias.to(dt))\n    r, nr = _rows_arg(rows)\n    nrows = nr if r is not None "
         "else len(cs) * m_local",
         "b = None if bias is None else _c(bias.to(torch.float16))\n    r, nr = _rows_arg(rows)\n    nrows = nr if r is "
         "not None else len(cs) * m_local")],
    "full-quant scales rounded to bf16": [
        ("        s_in = _c(x1_scale.float())", "        s_in = _c(x1_scale.to(torch.bfloat16).float())")],
}


def _run_pins(lib_path, package_dir=None):
    """Run the pins in a child process against the oracle library `lib_path`
    (and, with `package_dir`, the oracle package found there)."""
    env = dict(os.environ, MC2_ORACLE_LIB=lib_path, OMP_NUM_THREADS="2")
    args = [*PINS, "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider", "-p", "no:randomly"]
    if package_dir is None:
        cmd = [sys.executable, "-m", "pytest", *args]
    else:
        # import the copy first: the test modules then find it in sys.modules
        code = ("import sys; sys.path.insert(0, %r); import oracle; "
                "assert oracle.__file__.startswith(%r), oracle.__file__; "
                "import pytest; sys.exit(pytest.main(%r))" % (package_dir, package_dir, args))
        cmd = [sys.executable, "-c", code]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Build every mutant (and the unchanged copy) and run the pins against each, in parallel."""
    src = open(SRC).read()
    d = tmp_path_factory.mktemp("oracle_mutants")
    jobs = {"unchanged": src}
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, f"mutant '{name}': its text occurs {src.count(old)} times in the oracle"
        jobs[name] = src.replace(old, new)

    py_src = open(PY_SRC).read()
    py_jobs = {}
    for name, edits in PY_MUTANTS.items():
        text = py_src
        for old, new in edits:
            assert text.count(old) == 1, f"mutant '{name}': its text occurs {text.count(old)} times in the wrapper"
            text = text.replace(old, new)
        py_jobs[name] = text
    base_lib = oracle.compile_library(SRC, str(d / "libbase.so"))

    def one(item):
        i, (name, text) = item
        c = d / f"m{i}.c"
        c.write_text(text)
        lib = oracle.compile_library(str(c), str(d / f"libm{i}.so"))
        return name, _run_pins(lib)

    def one_py(item):
        i, (name, text) = item
        pkg = d / f"py{i}"
        (pkg / "oracle").mkdir(parents=True)
        (pkg / "oracle" / "__init__.py").write_text(text)
        return name, _run_pins(base_lib, str(pkg))

    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with ThreadPoolExecutor(workers) as ex:
        out = dict(ex.map(one, enumerate(jobs.items())))
        out.update(ex.map(one_py, enumerate(py_jobs.items())))
    return out


def test_unchanged_copy_passes_the_pins(outcomes):
    rc, log = outcomes["unchanged"]
    assert rc == 0, f"the pins fail on an unchanged copy of the oracle:\n{log}"


@pytest.mark.parametrize("name", list(MUTANTS) + list(PY_MUTANTS))
def test_pins_catch_the_planted_mistake(outcomes, name):
    rc, log = outcomes[name]
    # exit code 1: tests ran and at least one failed (not a collection or usage error)
    assert rc == 1 and "failed" in log, f"no pin caught the mutant '{name}' (pytest exit {rc}):\n{log}"
