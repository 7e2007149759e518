"""The parity suite's small shapes under device-side bounds checks.

The library is built a second time with MHA_BOUNDS_CHECK: in the attention
forward and backward kernels and in the projection and layer-norm GEMMs every
TMA coordinate and every direct global store is checked against the
problem's extents, and a failed check records MHA_ERR_BOUNDS in the status
word and skips the access.  The small-shape parity tests (ragged tails, both
key splits, every mask, MHA with and without layer normalisation, the
backward, the encoder layer) then run in a child process against that build:
each of them asserts a zero status word after its calls, and their outputs
must still match the oracle.  (The SIMT kernels -- decode, positional
encoding, fp32 attention -- take their indices from the grid and have no
status word; their stores are guarded by explicit range conditions.)"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# everything but the full-size workloads
SMALL = "not config5 and not configs_full and not config4_full and not workload_full"


def _checked_library():
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_tsds_build_checked", os.path.join(ROOT, "transformer_scaled_dot_softmax_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(checked=True)


def test_small_parity_cases_pass_with_bounds_checks():
    lib_path = _checked_library()
    env = dict(os.environ, MHA_LIBRARY=lib_path)
    probe = subprocess.run(
        [sys.executable, "-c",
         "from transformer_scaled_dot_softmax_gb300 import _native as n; print(n.LIB_PATH)"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr
    assert os.path.samefile(probe.stdout.strip(), lib_path)
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
         os.path.join("tests", "test_gpu_parity.py"), os.path.join("tests", "test_gpu_backward.py"),
         os.path.join("tests", "test_gpu_encoder.py"), "-k", SMALL],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-2000:])
    summary = [ln for ln in r.stdout.splitlines() if " passed" in ln]
    assert summary, r.stdout[-2000:]
    print("bounds-checked build:", summary[-1])
    import re
    assert int(re.search(r"(\d+) passed", summary[-1]).group(1)) >= 100
