"""The bounds-checked build (libgdn_debug.so, compiled with GDN_DEBUG_BOUNDS):
every global, shared-memory and TMEM index of the kernels is checked against
the extent of its buffer, and a failed check is recorded instead of trapping.

Two checks of it, each in a child process that selects the library with
GDN_DEBUG_BOUNDS=1:
  * its positive control trips exactly the three requests planted in it (and
    nothing else: the words are clear before and after);
  * the small parity cases of every kernel pass under it, while the binding
    reads the bounds words after every call and raises BoundsError on the
    first failed check, so every index those cases reach stayed in bounds.
"""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

# the parity files run under the checked build; the cases left out are the
# full-size ones (the 4 x 8192 prefill, 64-step decode loops) whose indices
# are those of the smaller cases at other sizes
PARITY_FILES = ["test_gpu_decode.py", "test_gpu_verify.py", "test_gpu_prefill.py", "test_gpu_kda.py",
                "test_gpu_kda_prefill.py", "test_gpu_slot_ops.py", "test_gpu_state_xfer.py", "test_gpu_epilogue.py",
                "test_gpu_mixed.py", "test_gpu_zero_decay.py", "test_zz_no_alloc.py"]
SKIP = "not four_by_8192 and not 64_steps and not 8192"


@pytest.fixture(scope="module")
def debug_lib(cuda):
    from hybrid_linear_attention_gdn_gb300 import _build
    return _build.build(debug_bounds=True)


def _child(args, timeout):
    env = dict(os.environ, GDN_DEBUG_BOUNDS="1")
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


POSITIVE_CONTROL = r"""
import torch
import hybrid_linear_attention_gdn_gb300 as gdn
from hybrid_linear_attention_gdn_gb300 import binding
assert gdn.debug_bounds() and binding.library_path().endswith("libgdn_debug.so")
torch.zeros(1, device="cuda")
assert gdn.debug_bounds_take() is None
gdn.selftest_bounds()
got = gdn.debug_bounds_take()
print(got)
count, where, index, limit = got
assert count == 3, got
assert where.startswith("slot_ops.cu:") and where.endswith(" global"), got
assert (index, limit) == (4, 4), got
assert gdn.debug_bounds_take() is None
print("positive control ok")
"""


def test_checked_build_positive_control(debug_lib):
    r = _child(["-c", POSITIVE_CONTROL], timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "positive control ok" in r.stdout


def test_normal_build_checks_nothing(cuda):
    import hybrid_linear_attention_gdn_gb300 as gdn
    from hybrid_linear_attention_gdn_gb300 import binding
    if binding.debug_bounds():
        pytest.skip("this process runs the checked build")
    lib = gdn.load()
    assert lib.gdn_selftest_bounds(None) == binding.ERR_UNSUPPORTED
    with pytest.raises(gdn.GdnError):
        gdn.debug_bounds_take()


def test_small_parity_cases_under_the_checked_build(debug_lib):
    files = [os.path.join("tests", f) for f in PARITY_FILES]
    r = _child(["-m", "pytest", *files, "-m", "gpu", "-k", SKIP, "-x", "-q", "-p", "no:cacheprovider"],
               timeout=2400)
    tail = r.stdout[-4000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert "BoundsError" not in r.stdout, tail
    # every selected case ran (128 at the time of writing), none skipped
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 120 and " skipped" not in r.stdout, tail
