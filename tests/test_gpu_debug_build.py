"""The bounds-checked build on the GPU.

libmala_debug.so is the same source compiled with -DMALA_DEBUG: every TMA box
origin and every global index of the tensor-core forward and backward and of
the decode kernel is checked against the extents the host validated before
the launch.  A failed check sets bit 8 of the device status word and skips
the access (a skipped load then ends in an expired, bounded wait), so nothing
faults.  The small parity cases run against it in a child process
(MALA_LIBRARY=debug); each of them asserts that the device status word is 0
after its calls, so a single out-of-range coordinate fails the run."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    "tests/test_gpu_prefill.py::test_tiny_fp32_workload",
    "tests/test_gpu_prefill.py::test_bf16_small_cases",
    "tests/test_gpu_prefill.py::test_bf16_gqa_small",
    "tests/test_gpu_prefill.py::test_bf16_batch2_gqa",
    "tests/test_gpu_prefill.py::test_bf16_noncausal",
    "tests/test_gpu_prefill.py::test_bf16_gradients_in_bf16",
    "tests/test_gpu_prefill.py::test_fp32_output_from_bf16_inputs",
    "tests/test_gpu_decode.py::test_decode_small_bf16",
    "tests/test_gpu_decode.py::test_decode_group_sizes",
    "tests/test_gpu_decode.py::test_decode_single_partial_tile",
    "tests/test_gpu_decode.py::test_decode_varlen_bf16",
    "tests/test_gpu_decode.py::test_decode_per_head_small_bf16",
    "tests/test_gpu_decode.py::test_decode_split_state_closed_form",
    "tests/test_gpu_varlen.py::test_varlen_bf16_ragged",
    "tests/test_gpu_varlen.py::test_varlen_bf16_gqa_and_bf16_grads",
    "tests/test_gpu_varlen.py::test_varlen_noncausal",
]


def test_small_parity_cases_pass_under_the_bounds_checked_build():
    from mass_adaptive_sparse_gb300 import build
    if not os.path.exists(build.LIB_DEBUG):
        build.build(variants=("debug",))
    env = dict(os.environ, MALA_LIBRARY="debug")
    probe = subprocess.run([sys.executable, "-c", "from mass_adaptive_sparse_gb300 import api; api.lib(); "
                            "print(api.LIB_PATH)"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libmala_debug.so"), probe.stdout + probe.stderr
    run = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *CASES],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert run.returncode == 0, run.stdout[-4000:] + run.stderr[-2000:]
    assert " passed" in run.stdout and "failed" not in run.stdout
