"""Planted mistakes in the oracle: each one must fail a pin (CPU only).

The pins in ``test_oracle_pins.py`` are worth what they catch.  Each case below copies the
oracle's C source, plants one plausible mistake in the copy (a dropped term, a wrong
bound, sign, index or tie rule, a transposed operand or layout), builds the copy with the
oracle's own compiler flags, and runs the pins against that build in a child process: the
pins must fail.  A control case runs them against an unchanged copy, built the same way,
and must pass, so that a failure means the planted mistake and not the harness.  The
oracle under ``oracle/`` is never changed.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "srkv_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# The child points the oracle package at the given build, then runs the pins, stopping at the
# first failure.
CHILD = (
    "import sys, oracle, pytest\n"
    "oracle.build = lambda force=False: sys.argv[1]\n"
    "sys.exit(pytest.main([sys.argv[2], '-x', '-q', '-p', 'no:cacheprovider']))\n")

# (name, text in the oracle's source, the planted replacement).  Every occurrence is replaced.
MUTANTS = [
    # attention: softmax(q K^T / sqrt(d)) V
    ("softmax scale dropped",
     "const double scale = 1.0 / sqrt((double)d);", "const double scale = 1.0;"),
    ("output not divided by the softmax denominator",
     "o[e] /= denom;", "o[e] /= 1.0;"),
    ("keys attended in place of values",
     "o[e] += w * kv_value(c, in, 1,", "o[e] += w * kv_value(c, in, 0,"),
    ("query heads of a group interleaved across kv heads",
     "const int64_t qh = h * G + j;", "const int64_t qh = h + j * Hkv;"),
    ("page layout read as [page][token][kv head][d]",
     "((page * Hkv + h) * S + t % S) * d + e", "((page * S + t % S) * Hkv + h) * d + e"),
    # the attended token set
    ("window starts one token late",
     "(t >= W) || selected[t / S]", "(t > W) || selected[t / S]"),
    ("one initial token too many",
     "attended[t] = (t < INIT)", "attended[t] = (t <= INIT)"),
    ("window one token short",
     "const int64_t W = L - LOCAL;", "const int64_t W = L - LOCAL + 1;"),
    # candidates, scores and the selection
    ("blocks that only touch the offload range are candidates",
     "return lo < hi;", "return lo <= hi;"),
    ("group query is its first head only",
     "for (int64_t j = 0; j < G; ++j)\n    for (int64_t e = 0; e < d; ++e)\n      qbar[e] +=",
     "for (int64_t j = 0; j < 1; ++j)\n    for (int64_t e = 0; e < d; ++e)\n      qbar[e] +="),
    ("partial block averaged over the whole block",
     "rep[e] = sum / (double)(last - first);", "rep[e] = sum / (double)S;"),
    ("block scores scaled by 1/sqrt(d)",
     "s += qbar[e] * rep[e];", "s += qbar[e] * rep[e] / sqrt((double)d);"),
    ("lowest scores kept",
     "if (a->score > b->score) return -1;\n  if (a->score < b->score) return 1;",
     "if (a->score > b->score) return 1;\n  if (a->score < b->score) return -1;"),
    ("ties go to the higher block",
     "return (a->block > b->block) - (a->block < b->block);",
     "return (a->block < b->block) - (a->block > b->block);"),
    ("kept count rounded down",
     "double x = ceil(p * (double)n - 1e-9);", "double x = floor(p * (double)n + 1e-9);"),
    ("kept count without the allowance for the binary error of p",
     "double x = ceil(p * (double)n - 1e-9);", "double x = ceil(p * (double)n);"),
    ("dense at the boundary itself",
     "const int dense = prompt < (int64_t)c->dense_boundary;",
     "const int dense = prompt <= (int64_t)c->dense_boundary;"),
    # prefill vectors and the footprint
    ("page vector averaged over the whole page",
     "rep[e] = v > 0 ? sum / (double)v : 0.0;", "rep[e] = v > 0 ? sum / (double)S : 0.0;"),
    ("footprint without K and V counted apart",
     "return 2.0 * batch * layers", "return batch * layers"),
    # E4M3 pages
    ("E4M3 exponent bias 8",
     "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("E4M3 subnormals one binade low",
     "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    ("E4M3 ties to the odd code",
     "(dist == bd && (code & 1u) == 0)", "(dist == bd && (code & 1u) == 1)"),
    ("row scale for a largest value of 240 (another 8-bit format's)",
     "amax / 448.0f", "amax / 240.0f"),
    ("quotient x / scale taken in double, not fp32",
     "const float y = (float)value_at(x, 0, e) / scale;",
     "const double y = value_at(x, 0, e) / (double)scale;"),
    ("NaN coded with the sign bit set",
     "if (isnan(x)) return 0x7fu;", "if (isnan(x)) return 0xffu;"),
    ("row scale indexed by element",
     "sc[i / c->head_dim]", "sc[i % c->head_dim]"),
]


def _build(folder, text: str) -> str:
    src = os.path.join(folder, "srkv_oracle.c")
    so = os.path.join(folder, "libsrkv_oracle.so")
    with open(src, "w") as f:
        f.write(text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", so, src, "-lm", "-lpthread"])
    return so


def _pins(so: str) -> subprocess.CompletedProcess:
    return subprocess.run([sys.executable, "-c", CHILD, so, PINS], cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


def _source() -> str:
    with open(SRC) as f:
        return f.read()


@pytest.fixture(scope="module")
def runs(tmp_path_factory):
    """Every copy (the unchanged one under None, then each planted mistake by name) built and
    run against the pins, several child processes at a time."""
    text = _source()
    for name, old, _ in MUTANTS:
        assert old in text, f"the text for {name!r} is not in the oracle's source"
    jobs = [(None, text)] + [(name, text.replace(old, new)) for name, old, new in MUTANTS]
    folders = [str(tmp_path_factory.mktemp(f"copy{i}")) for i in range(len(jobs))]

    def run(i):
        name, body = jobs[i]
        return name, _pins(_build(folders[i], body))

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as pool:
        return dict(pool.map(run, range(len(jobs))))


def test_pins_pass_on_an_unchanged_copy(runs):
    run = runs[None]
    assert run.returncode == 0, run.stdout[-2000:] + run.stderr[-2000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(runs, name):
    run = runs[name]
    # pytest's exit code 1: tests ran and at least one failed (not a collection or usage error).
    assert run.returncode == 1, (name, run.returncode, run.stdout[-2000:], run.stderr[-2000:])
    assert " failed" in run.stdout, (name, run.stdout[-2000:])
