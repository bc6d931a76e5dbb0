"""The debug build of the library (``libuaa_debug.so``, compiled with -DUAA_DEBUG).

In that build every kernel range-checks, before each access, the shared-memory
descriptors and TMEM addresses of its tensor-core operations (they must lie in
the CTA's own shared memory and TMEM allocation) and every output store of the
attention kernels (it must lie inside its tensor); a failed check skips the
access and makes ``check_device_status()`` raise UAA_ERR_DEBUG_CHECK.  This test
builds that library and re-runs the edge-case GPU tests -- ragged and single-row
tiles, interior and trailing masked key tiles, keyless batches, more than 256
mask rows, Sq != Sk, grouped launches, the masked exchange path, the fused
exchanges over uneven and empty shards, the one-pass backward, the canary
guard bands and tensors past 2^31 elements -- in a child process that loads
it: each of those tests checks the device status after its calls, so any failed
check fails it, and their parity checks must hold as in the release build.
"""
import os
import re
import subprocess
import sys

import pytest

import ulysses_dit_attention_gb300 as uaa

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD_SELECTION = [
    "tests/test_gpu_debug_build.py::test_loaded_library_is_the_debug_build",
    "tests/test_gpu_attention.py",
    "tests/test_gpu_fused_ulysses.py",
    "tests/test_gpu_fused_backward.py",
    "tests/test_gpu_guard_bands.py",
    "tests/test_gpu_large_offsets.py",
]
# the full-size workloads (sampled heads of S = 27280 and S = 4096) are left to the release run:
# they exercise the same kernels on more items, not other addressing
CHILD_DESELECT = "not 27k and not emulation_workload and not workload_sampled_heads"


def test_loaded_library_is_the_debug_build():
    if os.environ.get("UAA_DEBUG", "") != "1":
        pytest.skip("runs in the child process that loads the debug build")
    assert uaa.debug_build()
    assert "debug" in uaa.lib().uaa_version().decode()


def test_edge_cases_pass_the_debug_build_checks():
    from ulysses_dit_attention_gb300 import build

    build.build(debug=True)
    env = dict(os.environ, UAA_DEBUG="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "gpu", "-k", CHILD_DESELECT]
    r = subprocess.run(cmd + CHILD_SELECTION, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = "\n".join((r.stdout + r.stderr).strip().splitlines()[-30:])
    assert r.returncode == 0, f"edge cases under the debug build failed:\n{tail}"
    m = re.search(r"(\d+) passed", tail)
    # the marker test and the 60-odd edge-case tests all ran under the debug build
    assert m and int(m.group(1)) >= 60 and " failed" not in tail and " skipped" not in tail, tail
