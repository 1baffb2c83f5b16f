"""The bounds-checked build (libavsg_debug.so, compiled with
-DAVSG_DEBUG_BOUNDS): every index a kernel takes from the step's data or the
buffer state is checked against its array before the access, and a failure
is latched as AVSG_ERR_INTERNAL.  It stands in for a memory checker.  The
small parity workloads run through it in a child process (the library is
chosen once per process) -- overlapped and serial step orders, the no-reuse
path -- and must give the oracle's results with no check failing."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

SCRIPT = r"""
import sys
sys.path.insert(0, {tests!r})
import workload as W
from decode_serving_gb300 import avsg
from gpu_harness import ATTN_TOL, Parity
assert avsg.load_library()._name.endswith("libavsg_debug.so")
from test_gpu_parity import SMALL
for name in sorted(SMALL):
    for no_reuse in (False, True):
        p = Parity(SMALL[name], no_reuse=no_reuse)
        try:
            p.run()
            st = p.sess.stats()
            assert st.device_error == 0, (name, no_reuse, st.device_error, st.error_unit,
                                          st.error_position)
            if not no_reuse:
                assert st.hits == p.ref.hits and st.misses == p.ref.misses, name
            assert p.max_err <= ATTN_TOL, (name, p.max_err)
        finally:
            p.close()
print("bounds ok")
"""


@pytest.fixture(scope="module")
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_serving_gb300 import build
    return build.build(debug_bounds=True)


@pytest.mark.parametrize("overlap", ["1", "0"])
def test_small_workloads_pass_every_bounds_check(debug_lib, overlap):
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, AVSG_LIBRARY=debug_lib, AVSG_OVERLAP=overlap)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(tests=here)],
                       cwd=os.path.dirname(here), env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "bounds ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]
