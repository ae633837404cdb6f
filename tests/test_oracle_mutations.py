"""The oracle's pins catch plausible mistakes: each case below plants one
mistake in a temporary copy of ``oracle/`` (never in the oracle itself, and
on the CPU only) and runs the oracle's pin tests against that copy, which
must then fail.  The unchanged copy must pass.

Mistakes planted (one at a time):
  * x / s computed as x * (1/s) (the quotient's rounding, R2);
  * the UE8M0 exponent taken one lower (ceil vs floor of log2, R4);
  * codec ties rounded to the odd code instead of the even one;
  * the weight scales tiled instead of repeated over the n groups;
  * INT8 rounding half away from zero instead of half to even (R1);
  * the backward's W^T quantized in the other FP8 format than the one asked for;
  * the all-zero block clamp changed from 1e-10;
  * the subnormal exponent bias off by one;
  * block scales tiled instead of repeated along K.
"""
import os
import shutil
import subprocess
import sys

import pytest

from tests.conftest import ROOT

PIN_TESTS = ["tests/test_oracle_formats.py", "tests/test_oracle_quantize.py", "tests/test_oracle_gemm.py"]

MUTATIONS = {
    "reciprocal_division": ("quantize.py", "return (a64 / b64).astype(np.float32)",
                            "return (a64.astype(np.float32) * (np.float32(1.0) / b64.astype(np.float32)))"
                            ".astype(np.float32)"),
    "ue8m0_floor": ("quantize.py", "return np.where(m == 0.5, e - 1, e).astype(np.int64)",
                    "return (e - 1).astype(np.int64)"),
    "ties_to_odd": ("formats.py", "((d_hi == d_lo) & (codes[hi] % 2 == 0))",
                    "((d_hi == d_lo) & (codes[hi] % 2 == 1))"),
    "weight_scales_tiled": ("gemm.py", "sb_per_n = np.repeat(sb, group_n, axis=0)",
                            "sb_per_n = np.tile(sb, (group_n, 1))"),
    "int8_half_away": ("quantize.py", "return np.clip(np.rint(q.astype(np.float64)), -127, 127).astype(np.int8)",
                       "return np.clip(np.trunc(q.astype(np.float64) + np.copysign(0.5, q)), -127, 127)"
                       ".astype(np.int8)"),
    "backward_operand_format": ("gemm.py", 'wt, wt_s = mx_quantize(W, "rows", fp8)',
                                'wt, wt_s = mx_quantize(W, "rows", "e4m3" if fp8 == "e5m2" else "e5m2")'),
    "zero_block_clamp": ("quantize.py", "s = np.maximum(r, np.float32(1e-10)).astype(np.float32)",
                         "s = np.maximum(r, np.float32(1e-12)).astype(np.float32)"),
    "subnormal_bias": ("formats.py", "v = math.ldexp(m / (1 << fmt.man_bits), 1 - fmt.bias)",
                       "v = math.ldexp(m / (1 << fmt.man_bits), -fmt.bias)"),
    "block_scales_tiled": ("gemm.py", "return v * np.repeat(scales, bs, axis=-1)",
                           "return v * np.tile(scales, bs)"),
}


def _copy_tree(dst):
    for d in ("oracle", "workloads"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d), ignore=shutil.ignore_patterns("__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ["conftest.py", "__init__.py"] + [os.path.basename(t) for t in PIN_TESTS]:
        src = os.path.join(ROOT, "tests", f)
        if os.path.exists(src):
            shutil.copy(src, os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), dst)


def _run_pins(dst):
    env = dict(os.environ, PYTHONPATH=dst, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", *PIN_TESTS],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-600:]


def test_unchanged_copy_passes(tmp_path):
    _copy_tree(str(tmp_path))
    rc, out = _run_pins(str(tmp_path))
    assert rc == 0, out


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(tmp_path, name):
    _copy_tree(str(tmp_path))
    fname, old, new = MUTATIONS[name]
    path = os.path.join(str(tmp_path), "oracle", fname)
    src = open(path).read()
    assert src.count(old) == 1, f"{name}: the line to change is no longer in oracle/{fname}"
    open(path, "w").write(src.replace(old, new))
    rc, out = _run_pins(str(tmp_path))
    assert rc != 0, f"{name}: every pin still passes\n{out}"
