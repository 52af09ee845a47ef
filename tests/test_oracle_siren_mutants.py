"""The SIREN pins must catch plausible mistakes: each case plants one in a
copy of oracle/siren.py (loaded through HG_SIREN_ORACLE) and runs
tests/test_oracle_siren_pins.py against it, which has to fail; the
unmodified copy has to pass."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "siren.py")

# (name, original text, planted mistake)
MUTANTS = [
    ("Laplacian drops the squared-gradient term",
     "lapu = (-omega ** 2 * a * (y ** 2).sum(axis=1) + omega * c * s) @ W2.T", "lapu = (omega * c * s) @ W2.T"),
    ("Laplacian curvature-term sign", "lapu = (-omega ** 2 * a * (y ** 2)", "lapu = (omega ** 2 * a * (y ** 2)"),
    ("Laplacian drops omega on the lap-gamma term", "(y ** 2).sum(axis=1) + omega * c * s) @ W2.T",
     "(y ** 2).sum(axis=1) + c * s) @ W2.T"),
    ("gradient missing omega", "du = (omega * c[:, None, :] * y) @ W2.T", "du = (c[:, None, :] * y) @ W2.T"),
    ("value through cos", "u = a @ W2.T + b2", "u = c @ W2.T + b2"),
    ("backward: sine-layer derivative sign", "g_z = omega * c * g_a - omega * a * g_c",
     "g_z = omega * c * g_a + omega * a * g_c"),
    ("backward: squared term loses its 2", "- 2 * omega ** 2 * (a * P)[:, None, :] * y",
     "- omega ** 2 * (a * P)[:, None, :] * y"),
    ("backward: first-layer gradient pairs gamma with lap", "\"gW1\": g_z.T @ gamma", "\"gW1\": g_z.T @ lap"),
    ("backward: output bias from the Laplacian upstream", "\"gb2\": gu.sum(axis=0)", "\"gb2\": glu.sum(axis=0)"),
    ("backward: lap-gamma gradient without the cosine", "g_s = omega * c * P", "g_s = omega * P"),
    ("forward magnitudes ignore the input magnitudes", "mz = mg @ A(W1).T + A(b1)", "mz = A(gamma) @ A(W1).T + A(b1)"),
    ("forward magnitudes ignore the gradient-input magnitudes", "my = mdg @ A(W1).T\n        ms = ml",
     "my = A(dgamma) @ A(W1).T\n        ms = ml"),
]


def _pins_pass(path):
    env = dict(os.environ, HG_SIREN_ORACLE=path)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_siren_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    return r.returncode == 0, r.stdout[-400:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    from concurrent.futures import ThreadPoolExecutor
    with open(SRC) as f:
        source = f.read()
    d = tmp_path_factory.mktemp("siren_mutants")
    jobs = {"control": source}
    for name, orig, bad in MUTANTS:
        assert source.count(orig) == 1, f"mutation anchor for '{name}' not unique in siren.py"
        jobs[name] = source.replace(orig, bad)
    paths = {}
    for i, (name, text) in enumerate(jobs.items()):
        p = d / f"siren_m{i}.py"
        p.write_text(text)
        paths[name] = str(p)
    with ThreadPoolExecutor(max_workers=max(1, min(len(paths), os.cpu_count() or 2))) as ex:
        return dict(zip(paths, ex.map(_pins_pass, paths.values())))


def test_unmodified_copy_passes(outcomes):
    ok, out = outcomes["control"]
    assert ok, out


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(outcomes, name, orig, bad):
    ok, out = outcomes[name]
    assert not ok, f"the pins did not catch: {name}"
