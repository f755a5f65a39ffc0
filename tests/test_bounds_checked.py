"""The bounds-checking build (LA_CHECK_BOUNDS; build.py --checked): the same
sources with the tensor-core kernels' index checks compiled in, each failed
check recorded in the device error word (LA_ERR_BOUNDS) instead of an access.
Host-only here: it builds (the check macros compile for sm_103a), exports the
same entry points as the normal library, and reports itself through
la_build_flags; the normal library does not.  The GPU side runs in
tests/test_gpu_bounds_checked.py."""
import ctypes
import re
import subprocess

from linear_attention_head_gb300 import _native as N
from linear_attention_head_gb300 import build as libbuild


def _exports(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    return set(re.findall(r"\sT\s+(la_\w+)", out))


def test_checked_build_exports_the_same_entry_points_and_says_so():
    normal = libbuild.build()
    checked = libbuild.build(checked=True)
    assert checked != normal
    assert _exports(checked) == _exports(normal)
    lib_c = ctypes.CDLL(checked)
    lib_c.la_build_flags.restype = ctypes.c_int32
    assert lib_c.la_build_flags() & N.LA_BUILD_BOUNDS_CHECKED
    lib_n = ctypes.CDLL(normal)
    lib_n.la_build_flags.restype = ctypes.c_int32
    assert lib_n.la_build_flags() == 0
