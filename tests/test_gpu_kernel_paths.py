"""Every kernel family against the oracle, whatever the size heuristics pick:
the TMA-gather forward, the generic kernels, the specialised forward where
the generic one is chosen (small one-slot 16-bit problems), direct (unstaged)
parameter loads, the staged loads without the bulk copy, the backward's
corner merge forced on and off, ordinary (non-programmatic) launches, and
the FP32 accumulator on chip forced on (with tiles of 16 rows: most points
straddle tiles) and off, and the backward run one pass per level (with and
without the corner merge, with the touch classes of the FP32 workspace's
rows off, with every level or no level sparse, with four lanes a unit
instead of eight) or in one pass.  Each runs in a
child process with MSDA_TUNE set."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("tune", ["tma", "generic", "params=direct", "params=ld", "notma,P=1", "P=8", "pointparallel",
                                  "merge", "nomerge", "nopdl", "merge,P=2", "spec", "tiled", "tiled,tp=16", "notiled",
                                  "levelpass", "levelpass,merge", "nolevelpass", "levelpass,nomerge",
                                  "levelpass,notouch", "levelpass,tau=1", "levelpass,tau=1000", "levelpass,overlap",
                                  "levelpass,noc8", "levelpass,c8,notouch"])
def test_kernel_family(tune):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MSDA_TUNE=tune)
    r = subprocess.run([sys.executable, os.path.join(HERE, "path_parity_main.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
