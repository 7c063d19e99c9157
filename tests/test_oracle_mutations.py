"""The oracle's pins catch plausible mistakes: each case below plants one
mistake in a copy of oracle.c (on the CPU), and the pin suite
(tests/test_oracle.py) run against that copy must fail.  The mistakes are
the kind a reader checking the oracle against the pages would look for:
gate and up swapped, the bias subtracted, the tie-break reversed, a
coefficient of the gate-weight exp wrong, a block-scale index transposed,
the gate weight or the shared expert left out of the combine, E4M3 or bf16
rounding that truncates, an activation scale off by one step."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "gate_up_swapped": ("double hv = g / (1.0 + exp(-g)) * u;", "double hv = u / (1.0 + exp(-u)) * g;"),
    "bias_sign": ("if (b) acc += (double)b[e];", "if (b) acc -= (double)b[e];"),
    "tie_break_reversed": ("if (best < 0 || Lt[e] > Lt[best]) best = e;",
                           "if (best < 0 || Lt[e] >= Lt[best]) best = e;"),
    "exp_coefficient": ("c3 = (float)(1.0 / 6.0)", "c3 = (float)(1.0 / 6.5)"),
    "block_scale_transposed": (
        "g += pg * ((double)ev->sg[(int64_t)(i / QBLOCK) * HB + kb] * (double)sx[kb]);",
        "g += pg * ((double)ev->sg[(int64_t)kb * IB + (i / QBLOCK)] * (double)sx[kb]);"),
    "gate_weight_dropped": ("for (int32_t h = 0; h < H; ++h) acc[h] += wj * o[h];",
                            "for (int32_t h = 0; h < H; ++h) acc[h] += o[h];"),
    "e4m3_truncates": ("double m = nearbyint((ldexp(a, -E) - 1.0) * 8.0);",
                       "double m = floor((ldexp(a, -E) - 1.0) * 8.0);"),
    "quant_scale_off": ("? amax / 448.0f : 1.0f;", "? amax / 447.0f : 1.0f;"),
    "shared_expert_dropped": ("for (int32_t h = 0; h < H; ++h) acc[h] = o[h];",
                              "for (int32_t h = 0; h < H; ++h) acc[h] = 0.0 * o[h];"),
    "bf16_output_truncates": ("double r = nearbyint(a / ulp) * ulp;", "double r = floor(a / ulp) * ulp;"),
}


def run_pins_on(src: str, tmp_path):
    """Run tests/test_oracle.py against a mirror of the repository whose
    oracle is built from `src`; returns the completed process."""
    mirror = tmp_path / "root"
    (mirror / "oracle").mkdir(parents=True)
    for f in ("__init__.py", "oracle.h"):
        shutil.copy(os.path.join(ROOT, "oracle", f), mirror / "oracle" / f)
    (mirror / "oracle" / "oracle.c").write_text(src)
    os.symlink(os.path.join(ROOT, "synth"), mirror / "synth")
    (mirror / "tests").mkdir()
    for f in ("conftest.py", "test_oracle.py"):
        os.symlink(os.path.join(ROOT, "tests", f), mirror / "tests" / f)
    os.symlink(os.path.join(ROOT, "tests", "golden"), mirror / "tests" / "golden")
    env = dict(os.environ, PYTHONPATH=str(mirror))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        str(mirror / "tests" / "test_oracle.py")],
                       capture_output=True, text=True, timeout=600, cwd=str(mirror), env=env)
    # the pins ran on the mirror's build of the copy, not on the repository's oracle
    assert (mirror / "oracle" / "_oracle.so").exists(), r.stdout[-2000:] + r.stderr[-2000:]
    return r


def test_mirror_without_a_mistake_passes(tmp_path):
    """Control: the same mirror with the unchanged oracle (plus a comment, so
    it is rebuilt from the mirror's copy) passes every pin."""
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read() + "\n/* mirror copy */\n"
    r = run_pins_on(src, tmp_path)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_a_planted_mistake(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    old, new = MUTATIONS[name]
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert src.count(old) == 1, f"mutation site of {name} not found once"
    r = run_pins_on(src.replace(old, new), tmp_path)
    assert r.returncode != 0, f"no pin caught the mistake {name}:\n{r.stdout[-1500:]}"
    assert "1 failed" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]      # a pin failed, not a build error
