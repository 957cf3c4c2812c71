"""Rows-per-call statistics on the GPU: each successful verify call counts
once under its M (per plan, per active grouped problem, and for the process);
failed calls and the plan's launch measurement do not count; reset clears a
plan's or group's counts only; and LBV_VERIFY_STATS=1 prints the process's
counts at exit."""
import os
import subprocess
import sys

import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
K, N = 512, 256


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()


def operands(fmt, group, seed):
    spec = {lbv.FMT_SIGN1_G128: synth.SIGN1_G128, lbv.FMT_AFFINE2: synth.AFFINE2}[fmt]
    mat = synth.Matrix("rows", spec, K, N, group, "f16")
    parts, xb = synth.gen_matrix(mat, seed)
    Wp = torch.from_numpy(lbv.pack(fmt, parts, K, N, group)).cuda()
    X = torch.from_numpy(xb.view(np.int16)).cuda()
    return Wp, X


def hist(**counts):
    h = {m: 0 for m in range(1, 9)}
    for k, v in counts.items():
        h[int(k[1:])] = v
    return h


def test_plan_counts():
    Wp, X = operands(lbv.FMT_SIGN1_G128, 128, 3)
    before = lbv.rows_histogram()
    P = lbv.Plan(lbv.FMT_SIGN1_G128, K, N, 128, lbv.F16, lbv.PLAN_PDL | lbv.PLAN_MEASURE)
    assert P.rows_histogram() == hist()                  # the measurement is not counted
    Y = torch.zeros((8, N), dtype=torch.float32, device="cuda")
    for M in (1, 3, 3, 8):
        lbv.verify_gemm(P, X, M, Wp, Y)
    with pytest.raises(lbv.LbvError):
        lbv.verify_gemm(P, X, 9, Wp, Y)                  # rejected: not counted
    torch.cuda.synchronize()
    assert P.rows_histogram() == hist(m1=1, m3=2, m8=1)

    H = lbv.Plan(lbv.FMT_AFFINE2, K, N, 128, lbv.F16, lbv.PLAN_PDL)
    ws = torch.zeros(lbv.fused_workspace_bytes(), dtype=torch.uint8, device="cuda")
    idx = torch.zeros(8, dtype=torch.int32, device="cuda")
    Wa, Xa = operands(lbv.FMT_AFFINE2, 128, 4)
    lbv.verify_fused(H, Xa, 5, Wa, lbv.FUSED_ROTATE | lbv.FUSED_ARGMAX, idx=idx, workspace=ws)
    lbv.verify_fused(H, Xa, 5, Wa, lbv.FUSED_ROTATE, Y=Y)
    torch.cuda.synchronize()
    assert H.rows_histogram() == hist(m5=2)
    assert P.rows_histogram() == hist(m1=1, m3=2, m8=1)  # counts are per plan

    after = lbv.rows_histogram()
    assert {m: after[m] - before[m] for m in after} == hist(m1=1, m3=2, m5=2, m8=1)
    P.rows_reset()
    assert P.rows_histogram() == hist()
    assert lbv.rows_histogram() == after                 # the process counts stay
    P.close()
    H.close()


def test_group_counts():
    shapes = [(K, N), (K, N), (K, N)]
    G = lbv.Group(lbv.FMT_SIGN1_G128, 128, lbv.F16, shapes, lbv.PLAN_PDL)
    ops = [operands(lbv.FMT_SIGN1_G128, 128, 10 + i) for i in range(3)]
    Ys = [torch.zeros((8, N), dtype=torch.float32, device="cuda") for _ in shapes]
    before = lbv.rows_histogram()
    for Ms in ([2, 0, 7], [2, 2, 0], [0, 0, 0]):
        lbv.verify_grouped(G, [(X, M, W, Y) for (W, X), M, Y in zip(ops, Ms, Ys)])
    with pytest.raises(lbv.LbvError):
        lbv.verify_grouped(G, [(ops[0][1], 9, ops[0][0], Ys[0]), (None, 0, None, None),
                               (None, 0, None, None)])
    torch.cuda.synchronize()
    assert G.rows_histogram() == hist(m2=3, m7=1)
    after = lbv.rows_histogram()
    assert {m: after[m] - before[m] for m in after} == hist(m2=3, m7=1)
    G.rows_reset()
    assert G.rows_histogram() == hist()
    G.close()


CHILD = """
import numpy as np, torch
import few_row_packed_gb300 as lbv
import synth
K, N = 512, 256
mat = synth.Matrix("rows", synth.SIGN1_G128, K, N, 128, "f16")
parts, xb = synth.gen_matrix(mat, 3)
Wp = torch.from_numpy(lbv.pack(lbv.FMT_SIGN1_G128, parts, K, N, 128)).cuda()
X = torch.from_numpy(xb.view(np.int16)).cuda()
Y = torch.zeros((8, N), dtype=torch.float32, device="cuda")
P = lbv.Plan(lbv.FMT_SIGN1_G128, K, N, 128, lbv.F16, lbv.PLAN_PDL)
for M in (4, 4, 6):
    lbv.verify_gemm(P, X, M, Wp, Y)
torch.cuda.synchronize()
"""


def test_report_at_exit_after_calls():
    env = dict(os.environ, LBV_VERIFY_STATS="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("lbv: verify rows per call:")]
    assert lines == ["lbv: verify rows per call: 1:0 2:0 3:0 4:2 5:0 6:1 7:0 8:0 "
                     "(calls 3, mean rows 4.67)"]
