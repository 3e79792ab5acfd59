"""The debug build (libfa_gb300_debug.so, compiled with -DFA_DEBUG).

Its kernels check every global store's index against the buffer they were
given and record FA_ERR_DEBUG_CHECK instead of writing outside it.  A
cross-section of the GPU parity tests runs against it in a child process
(the binding loads the library named by FA_LIBRARY): the results must still
match the oracle, and the tests' device-status checks require every bounds
check to stay silent on valid inputs.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    "tests/test_gpu_bf16.py::test_small_shapes",
    "tests/test_gpu_bf16.py::test_varlen_small_full",
    "tests/test_gpu_bf16.py::test_varlen_causal_unequal_q_and_k_lengths",
    "tests/test_gpu_fp32.py",
    "tests/test_gpu_fp8.py",
    "tests/test_gpu_paged_prefill.py::test_paged_prefill_small",
    "tests/test_gpu_decode.py::test_decode_small_ragged",
    "tests/test_gpu_decode.py::test_split_combine_against_oracle_merge",
    "tests/test_gpu_decode.py::test_gathered_rows_equal_host_gather",
]

CHILD = """
import sys
import pytest
from tiled_online_softmax_sm_gb300 import binding as fb
lib = fb.load()
assert lib._name == sys.argv[1], (lib._name, sys.argv[1])
sys.exit(pytest.main(["-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"] + sys.argv[2:]))
"""


def test_debug_build_passes_parity_cases():
    from tiled_online_softmax_sm_gb300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, FA_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", CHILD, lib] + CASES, cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
