"""The pins must catch plausible mistakes.  Each case plants one mistake in a
copy of oracle/hg_oracle.c (on the CPU), builds it, and runs the pin suite
against it through HG_ORACLE_LIB; the suite has to fail.  The unmodified
source has to pass (a control, so a broken harness cannot pass vacuously)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "hg_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("drop dx^|alpha| scaling", "scale[k] = pow(dx, (double)k);   /* dx^{|alpha|} */\n    /* bases",
     "scale[k] = 1.0;   /* dx^{|alpha|} */\n    /* bases"),
    ("slope-basis derivative sign", "out[1] = (1.0 - a) * (1.0 - 3.0 * a);", "out[1] = (1.0 - a) * (1.0 + 3.0 * a);"),
    ("value-basis second derivative", "out[2] = -6.0 + 12.0 * a;", "out[2] = -6.0 + 6.0 * a;"),
    ("gradient missing the N factor", "if (dgamma) dgamma[j * F + f] += th * scale[k] * N * dH[j];",
     "if (dgamma) dgamma[j * F + f] += th * scale[k] * dH[j];"),
    ("Laplacian keeps one axis", "if (lap) lap[f] += th * scale[k] * N * N * d2H[j];",
     "if (lap && j == 0) lap[f] += th * scale[k] * N * N * d2H[j];"),
    ("one-sided direction ignored", "hermite_1d(a, t[i] - (double)vi, vi ? -1.0 : 1.0, hb[i][vi][a]);\n    for (int v = 0; v < (1 << d); ++v) {\n        int64_t g[OR_MAXD];\n        for (int i = 0; i < d; ++i) g[i] = c[i] + (v >> i & 1);     /* corner vertex */",
     "hermite_1d(a, t[i] - (double)vi, 1.0, hb[i][vi][a]);\n    for (int v = 0; v < (1 << d); ++v) {\n        int64_t g[OR_MAXD];\n        for (int i = 0; i < d; ++i) g[i] = c[i] + (v >> i & 1);     /* corner vertex */"),
    ("dense index axes transposed", "for (int i = 0; i < d; ++i) { idx += (uint64_t)g[i] * mul; mul *= side; }",
     "for (int i = 0; i < d; ++i) { idx += (uint64_t)g[d - 1 - i] * mul; mul *= side; }"),
    ("wrong hash prime", "{1u, 2654435761u, 805459861u, 3674653429u}", "{1u, 2654435769u, 805459861u, 3674653429u}"),
    ("wrong fourth hash prime", "805459861u, 3674653429u}", "805459861u, 3674653431u}"),
    ("hash adds instead of XOR", "h ^= (uint32_t)(((uint64_t)g[i] * OR_PRIMES[i]) & 0xffffffffu);",
     "h += (uint32_t)(((uint64_t)g[i] * OR_PRIMES[i]) & 0xffffffffu);"),
    ("colliding gradients overwrite", "gk[f] += w;", "gk[f] = w;"),
    ("slot order inside a bucket", "if (less) slot++;", "if (!less && lists[j][0] != mine[0]) slot++;"),
    ("d-linear weights swapped", "w *= vi ? t[i] : 1.0 - t[i];\n                }\n                uint32_t idx = vertex_index(d, g, res[l], log2T);\n                const double* th",
     "w *= vi ? 1.0 - t[i] : t[i];\n                }\n                uint32_t idx = vertex_index(d, g, res[l], log2T);\n                const double* th"),
    ("cell not clamped at x = 1", "if (ci > (int64_t)N - 1) ci = (int64_t)N - 1;\n    *c = ci;", "*c = ci;"),
    ("mixed second derivative drops one factor",
     "else hij *= (m == i || m == j) ? (*h[m])[1] : (*h[m])[0];",
     "else hij *= (m == i) ? (*h[m])[1] : (*h[m])[0];"),
    ("Hessian missing N^2", "hess[q * F + f] += th * scale[k] * N * N * hij;", "hess[q * F + f] += th * scale[k] * N * hij;"),
    ("FD shift directions swapped", "(j % 2 == 0) ? x[i] + eps : x[i] - eps;", "(j % 2 == 0) ? x[i] - eps : x[i] + eps;"),
    ("FD gradient over eps instead of 2 eps", "if (dgamma) dgamma[od] = (gp - gm) / (2.0 * e);",
     "if (dgamma) dgamma[od] = (gp - gm) / e;"),
    ("FD Laplacian drops the centre term", "lp += (gp - 2.0 * gs[0][f] + gm) / (e * e);", "lp += (gp + gm) / (e * e);"),
    ("FD backward centre weight without d", "u[0][f] = gg - 2.0 * d * gl / (e * e);", "u[0][f] = gg - 2.0 * gl / (e * e);"),
    ("FD backward stencil sign", "u[1 + j][f] = dir * gd / (2.0 * e) + gl / (e * e) + gs;",
     "u[1 + j][f] = gd / (2.0 * e) + gl / (e * e) + gs;"),
    ("RBF distance in x units", "y[i] = (double)c[i] + t[i];", "y[i] = ((double)c[i] + t[i]) / (double)N;"),
    ("RBF ring box shifted by one", "g[i] = c[i] - rings + 1 + rem % side;", "g[i] = c[i] - rings + rem % side;"),
    ("RBF weights not normalised", "const double w = phi[q] / S;", "const double w = phi[q];"),
    ("RBF Laplacian drops the cross term", "nb->lw[q] = Nd * Nd * (lphi[q] - 2.0 * dot - w * lS) / S;",
     "nb->lw[q] = Nd * Nd * (lphi[q] - w * lS) / S;"),
    ("RBF kernel derivative sign", "dphi[q][i] = -2.0 * e2 * (y[i] - (double)g[i]) * phi[q];",
     "dphi[q][i] = 2.0 * e2 * (y[i] - (double)g[i]) * phi[q];"),
    ("Hessian backward uses the pure derivative for mixed entries",
     "else x *= (m == i || m == j) ? (*h[m])[1] : (*h[m])[0];",
     "else x *= (m == i || m == j) ? (*h[m])[2] : (*h[m])[0];"),
]


def _build(src_text, out_dir, tag):
    c = os.path.join(out_dir, f"mut_{tag}.c")
    so = os.path.join(out_dir, f"libmut_{tag}.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-w",
                           "-o", so, c, "-lm"])
    return so


def _pins_pass(lib_path):
    env = dict(os.environ, HG_ORACLE_LIB=lib_path)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_hessian_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_fd_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_rbf_pins.py"), "-x", "-q", "-p",
                        "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    return r.returncode == 0, r.stdout[-400:]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.fixture(scope="module")
def outcomes(source, tmp_path_factory):
    """Build the control and every mutant, and run their pin suites
    concurrently (each in its own process): {name: (passed, tail of output)}."""
    from concurrent.futures import ThreadPoolExecutor
    d = str(tmp_path_factory.mktemp("mutants"))
    jobs = {"control": source}
    for i, (name, orig, bad) in enumerate(MUTANTS):
        assert source.count(orig) == 1, f"mutation anchor for '{name}' not unique in hg_oracle.c"
        jobs[name] = source.replace(orig, bad)
    libs = {name: _build(text, d, f"m{i}") for i, (name, text) in enumerate(jobs.items())}
    with ThreadPoolExecutor(max_workers=max(1, min(len(libs), os.cpu_count() or 2))) as ex:
        res = dict(zip(libs, ex.map(_pins_pass, libs.values())))
    return res


def test_unmodified_copy_passes(outcomes):
    ok, out = outcomes["control"]
    assert ok, out


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(outcomes, name, orig, bad):
    ok, out = outcomes[name]
    assert not ok, f"the pins did not catch: {name}"
