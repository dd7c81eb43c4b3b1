"""Planted mistakes in the oracle, on the CPU.

Each mutant is a copy of ``oracle/oracle.c`` with one plausible error written
into it: a dropped term, a wrong sign, index or operand order, a missing clip
or check. It is compiled on its own, with the oracle's own flags, and the pins
of its part of the oracle run against it. Every mutant must make at least one
pin fail, which shows that the pins tie the oracle to the pages' definitions
and to the mathematics rather than to its own code. An unmutated copy, built
and run the same way, must pass, so that a failure means the planted mistake.

The mutated copies are built in a scratch folder beside this file
(``tests/_mutants/``, ignored by git), which the test removes when it ends;
the oracle itself is never touched.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.c")

PINS = "test_oracle_pins.py"
PLANNER = "test_oracle_planner.py"
RING = "test_oracle_ring.py"
RDA = "test_oracle_rda.py"

# (what the mistake is, text in oracle.c, text put in its place, pins that must catch it)
MUTANTS = [
    ("pseudo-gradient sign flipped",
     "return theta_g - theta_k;", "return theta_k - theta_g;", PINS),
    ("non-finite values not counted",
     "if (!isfinite(d)) ++bad;", ";", PINS),
    ("mean accumulated in fp32",
     "double sum = 0.0;", "float sum = 0.0f;", PINS),
    ("sample sigma in place of the population sigma",
     "sqrt(ss / (double)n)", "sqrt(ss / (double)(n - 1))", PINS),
    ("clip range drops the mean",
     "lo[o] = mu - clip_sigmas * sigma;", "lo[o] = -clip_sigmas * sigma;", PINS),
    ("clip multiplier ignored on the upper edge",
     "hi[o] = mu + clip_sigmas * sigma;", "hi[o] = mu + 3.0 * sigma;", PINS),
    ("bucket index rounded instead of floored",
     "int b = (int)floor(u);", "int b = (int)floor(u + 0.5);", PINS),
    ("upper clip missing from the bucket mean",
     "if (v > H) v = H;", ";", PINS),
    ("empty bucket decodes to its lower edge",
     "((double)j + 0.5) * (H - L)", "((double)j) * (H - L)", PINS),
    ("degenerate range decodes to zero",
     "for (int j = 0; j < NB; ++j) cb[j] = (float)mean[o];",
     "for (int j = 0; j < NB; ++j) cb[j] = 0.0f;", PINS),
    ("negative weights accepted",
     "if (!(w >= 0.0) || !isfinite(w)) return OR_ERR_ARG;", ";", PINS),
    ("minimum quorum not enforced",
     "if (n_present < need) return OR_ERR_QUORUM;", ";", PINS),
    ("weights not normalised",
     "w_hat[k] = (float)(w / total);", "w_hat[k] = (float)w;", PINS),
    ("codebook indexed tensor-major",
     "\n                    v = codebook[((int64_t)k * T + t) * NB + codes[k][i]];",
     "\n                    v = codebook[((int64_t)t * K + k) * NB + codes[k][i]];", PINS),
    ("absent learners read by the merge",
     "                if (present && !present[k]) continue; /* absent: never read */\n"
     "                float v;",
     "                float v;", PINS),
    ("momentum operands transposed",
     "\n            float m_new = fmaf(mu, momentum[i], acc);",
     "\n            float m_new = fmaf(mu, acc, momentum[i]);", PINS),
    ("plain momentum in place of Nesterov",
     "\n            float g = fmaf(mu, m_new, acc);", "\n            float g = m_new;", PINS),
    ("outer learning rate with the wrong sign",
     "\n            float th = fmaf(-lr, g, theta_g[i]);",
     "\n            float th = fmaf(lr, g, theta_g[i]);", PINS),
    ("planner sorts the tensors ascending",
     "return x->numel > y->numel ? -1 : 1;", "return x->numel < y->numel ? -1 : 1;", PLANNER),
    ("planner fills the fullest fragment",
     "if (frag_load[p] < frag_load[best]) best = p;",
     "if (frag_load[p] > frag_load[best]) best = p;", PLANNER),
    ("ring hop adds the partial sum without re-quantising it",
     "cb[(int64_t)t * NB + code[i]]);", "P[i]);", RING),
    ("ring's first hop unweighted",
     "P[i] = w_hat[k] * pseudo_grad(", "P[i] = 1.0f * pseudo_grad(", RING),
    ("RDA radial part unweighted",
     "r += (double)w_hat[k] * nrm[k];", "r += nrm[k];", RDA),
    ("RDA directions not made unit vectors",
     "coef[k] = nrm[k] > 0.0 ? (double)w_hat[k] / nrm[k] : 0.0;",
     "coef[k] = (double)w_hat[k];", RDA),
    ("RDA scale ignores the length of the mean direction",
     "const double scale = uu > 0.0 ? r / sqrt(uu) : 0.0;", "const double scale = r;", RDA),
]

CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]


def _run_pins(workdir, tag, source, pins):
    """Builds `source` as a library and runs the `pins` file against it in a
    fresh interpreter; returns (pytest exit code, first failing test)."""
    c = os.path.join(workdir, f"{tag}.c")
    so = os.path.join(workdir, f"lib{tag}.so")
    with open(c, "w") as fh:
        fh.write(source)
    subprocess.run(["gcc", *CFLAGS, "-o", so, c, "-lm"], check=True)
    # the pins load the oracle through oracle.lib(), which takes the library
    # oracle.build() returns: point it at the mutant
    code = (
        "import sys\n"
        f"sys.path[:0] = [{ROOT!r}, {HERE!r}]\n"
        "import oracle\n"
        f"oracle.build = lambda force=False: {so!r}\n"
        "import pytest\n"
        f"sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', '--rootdir', {ROOT!r},"
        f" {os.path.join(HERE, pins)!r}]))\n"
    )
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       cwd=workdir, timeout=600)
    failed = [ln.split("::", 1)[-1] for ln in r.stdout.splitlines() if ln.startswith("FAILED")]
    return r.returncode, (failed[0] if failed else r.stdout[-400:])


def test_every_planted_mistake_fails_a_pin():
    workdir = os.path.join(HERE, "_mutants", str(os.getpid()))
    os.makedirs(workdir, exist_ok=True)
    try:
        _planted_mistakes(workdir)
    finally:
        shutil.rmtree(workdir, ignore_errors=True)
        try:
            os.rmdir(os.path.dirname(workdir))
        except OSError:
            pass


def _planted_mistakes(workdir):
    with open(SRC) as fh:
        src = fh.read()
    jobs = {"control": (src, PINS)}
    for i, (what, old, new, pins) in enumerate(MUTANTS):
        # each planted text must still name exactly one place in the oracle
        assert src.count(old) == 1, (what, src.count(old))
        jobs[f"m{i:02d}"] = (src.replace(old, new), pins)
    workers = max(2, min(8, os.cpu_count() or 2))
    with cf.ThreadPoolExecutor(workers) as ex:
        futs = {tag: ex.submit(_run_pins, workdir, tag, s, p) for tag, (s, p) in jobs.items()}
        res = {tag: f.result() for tag, f in futs.items()}
    rc, info = res.pop("control")
    assert rc == 0, f"the unmutated oracle fails its own pins: {info}"
    survivors = []
    for i, (what, _, _, pins) in enumerate(MUTANTS):
        rc, info = res[f"m{i:02d}"]
        if rc == pytest.ExitCode.TESTS_FAILED:
            print(f"{what}: caught by {info}")
        else:
            survivors.append((what, pins, rc, info))
    assert not survivors, survivors
