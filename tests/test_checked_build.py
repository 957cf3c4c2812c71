"""CPU tests of the checked build (liblbv_checked.so, compiled with
LBV_CHECKED): it builds, exports exactly the entry points include/lbv.h
declares, reports itself through lbv_checked_build (the release library
reports 0), and the binding loads it only when LBV_LIBRARY=checked."""
import os
import re
import subprocess
import sys

import pytest

from few_row_packed_gb300 import buildlib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lbv.h")


@pytest.fixture(scope="module")
def libs():
    return buildlib.build(), buildlib.build(checked=True)


def exported(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    return set(re.findall(r" T (lbv_\w+)", out))


def test_same_entry_points(libs):
    release, checked = libs
    declared = set(re.findall(r"^LBV_API [^(]*?\b(lbv_\w+)\(", open(HEADER).read(), re.M))
    assert "lbv_checked_build" in declared
    assert exported(release) == declared
    assert exported(checked) == declared


@pytest.mark.parametrize("env,flag", [(None, 0), ("checked", 1)])
def test_binding_selects_library(libs, env, flag):
    e = dict(os.environ)
    e.pop("LBV_LIBRARY", None)
    if env is not None:
        e["LBV_LIBRARY"] = env
    code = ("import few_row_packed_gb300 as lbv, os; "
            "print(os.path.basename(lbv.LIB_PATH), lbv.lib().lbv_checked_build())")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=e, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    name = "liblbv_checked.so" if flag else "liblbv.so"
    assert r.stdout.split() == [name, str(flag)]
