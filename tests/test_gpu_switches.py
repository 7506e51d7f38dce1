"""The documented environment switches select other code paths of the same
operations; each must give results that pass the same parity tests.

  WS_NF4_PAIR_MMA=0  two-CTA pairs copy the weight halves and issue one MMA
                     per CTA instead of one pair MMA
  WS_NF4_PDL=0       plain stream-ordered launches (no programmatic
                     dependent launch; the dequant GEMM launches cooperatively)
  WS_NF4_SIDE=0      the backward's dB stays on the caller's stream

A switch is read once per process, so each runs the linear parity tests
(which cover the pair kernels at M > 256 and the full-size shapes) and the
stack's recompute / streamed-equals-resident / graph tests in a child
pytest with the switch set."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SELECT = [
    "tests/test_gpu_linear.py::test_linear_fwd_bwd_parity",
    "tests/test_gpu_linear.py::test_full_size_sampled_rows",
    "tests/test_gpu_linear.py::test_nf4_matmul_alone",
    "tests/test_gpu_stack.py::test_recompute_backward_equals_saved_backward",
    "tests/test_gpu_stack.py::test_one_step_matches_oracle",
    "tests/test_gpu_stack.py::test_graph_replay_equals_eager",
]


@pytest.mark.parametrize("switch", ["WS_NF4_PAIR_MMA", "WS_NF4_PDL", "WS_NF4_SIDE"])
def test_switch_passes_parity(switch):
    env = dict(os.environ)
    env[switch] = "0"
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "gpu", *SELECT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, (switch, r.stdout[-3000:], r.stderr[-2000:])
