"""The bounds-checked debug build (compiled with -DRF_CHECK_BOUNDS).

Every kernel of that build checks each global index it computes against the
extent of its buffer, derived from the call's sizes; a refused index skips
its access and records RF_ERR_BOUNDS, which rf_device_error reports (no trap,
no fault).  Here:
  * the default library says it has no checks, and refuses the self-test;
  * the checked library's self-test presents one index past the end to the
    check and the status comes back (the store it guards targets a valid
    address either way);
  * the whole GPU parity suite runs again against the checked library, with
    an assertion after every test that no index was refused.
"""

import ctypes
import os
import subprocess
import sys

import pytest

from conftest import ROOT, load_builder


def test_default_build_has_no_checks():
    import cascaded_reductions_gb300 as rf
    if os.environ.get("RF_LIBRARY"):
        pytest.skip("another library was requested")
    assert rf.rf_bounds_checked() is False
    # refused on the host before any CUDA call
    assert rf._lib.rf_selftest_bounds(None) == rf.RF_ERR_UNSUPPORTED


@pytest.fixture(scope="module")
def checked_lib_path():
    return load_builder().build_checked()


@pytest.mark.gpu
def test_selftest_refused_index_is_reported(checked_lib_path):
    import cascaded_reductions_gb300 as rf
    lib = rf.load_library(checked_lib_path)
    assert lib.rf_bounds_checked() == 1
    st = ctypes.c_int(-1)
    assert lib.rf_device_error(ctypes.byref(st), None) == rf.RF_OK
    assert st.value == rf.RF_OK
    assert lib.rf_selftest_bounds(None) == rf.RF_OK
    assert lib.rf_device_error(ctypes.byref(st), None) == rf.RF_OK
    assert st.value == rf.RF_ERR_BOUNDS
    assert lib.rf_device_error(ctypes.byref(st), None) == rf.RF_OK
    assert st.value == rf.RF_OK                       # read and cleared


@pytest.mark.gpu
def test_parity_suite_refuses_no_index(checked_lib_path):
    env = dict(os.environ, RF_LIBRARY=checked_lib_path)
    cmd = [sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-x", "-q",
           "-p", "no:cacheprovider", "--ignore", os.path.join("tests", os.path.basename(__file__))]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = r.stdout[-4000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
