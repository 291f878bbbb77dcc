"""The checked build: the same sources compiled with -DTV_CHECKED=1, whose
device code tests index ranges before the accesses they guard and records
TV_ERR_BOUNDS instead of trapping (a stand-in for a memory checker, which
cannot run on every GPU machine).  This CPU test builds it into a temporary
folder, loads it, and checks that it reports itself as checked while the
normal build does not."""
import ctypes

import pytest

from speculative_decoding_tree_masked_gb300 import _build


def test_checked_build_compiles_links_and_says_so(tmp_path):
    try:
        _build._nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    lib_path = _build.build(extra_flags=["-DTV_CHECKED=1"], build_dir=str(tmp_path / "objs"),
                            lib_path=str(tmp_path / "libtreeverify_checked.so"))
    checked = ctypes.CDLL(lib_path)
    checked.tv_checked_build.restype = ctypes.c_int32
    assert checked.tv_checked_build() == 1
    checked.tv_status_string.restype = ctypes.c_char_p
    assert checked.tv_status_string(7) == b"device bounds check failed"
    # the normal build (incremental: only what changed is recompiled)
    normal = ctypes.CDLL(_build.build())
    normal.tv_checked_build.restype = ctypes.c_int32
    assert normal.tv_checked_build() == 0
