"""CPU tests of the rows-per-call statistics ("dflash-mlx-bonsai2" README,
Commands: a histogram of the drafted rows per verify call, printed at exit on
request): the calls reject NULL arguments, the process-wide counts start at
zero, and LBV_VERIFY_STATS controls the one-line report at exit."""
import ctypes
import os
import subprocess
import sys

import pytest

import few_row_packed_gb300 as lbv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    lbv.build()
    return lbv.lib()


def test_null_arguments(L):
    c = (ctypes.c_uint64 * 8)()
    assert L.lbv_rows_histogram(None) == lbv.ERR_INVALID_ARG
    assert L.lbv_plan_rows_histogram(None, c) == lbv.ERR_INVALID_ARG
    assert L.lbv_plan_rows_reset(None) == lbv.ERR_INVALID_ARG
    assert L.lbv_group_rows_histogram(None, c) == lbv.ERR_INVALID_ARG
    assert L.lbv_group_rows_reset(None) == lbv.ERR_INVALID_ARG
    assert "NULL" in lbv.last_error()


def run_child(env_value):
    env = dict(os.environ)
    env.pop("LBV_VERIFY_STATS", None)
    if env_value is not None:
        env["LBV_VERIFY_STATS"] = env_value
    code = ("import few_row_packed_gb300 as lbv; h = lbv.rows_histogram(); "
            "assert h == {m: 0 for m in range(1, 9)}, h")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return [ln for ln in r.stderr.splitlines() if ln.startswith("lbv: verify rows per call:")]


def test_report_at_exit(L):
    lines = run_child("1")
    assert lines == ["lbv: verify rows per call: 1:0 2:0 3:0 4:0 5:0 6:0 7:0 8:0 "
                     "(calls 0, mean rows 0.00)"]


@pytest.mark.parametrize("value", [None, "0", ""])
def test_no_report_unless_asked(L, value):
    assert run_child(value) == []
