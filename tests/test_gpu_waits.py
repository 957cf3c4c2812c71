"""Bounded waits that run out, on the GPU, without a fault: a plan made with
LBV_PLAN_TEST_WAIT_LIMIT gives its main-loop weight waits 256 tries and has
the first warp of the first CTA leave one weight copy out, so that warp's wait
gives up.  The warp must stop, let its issued copies land and the kernel end;
the plan's device status must report LBV_ERR_TIMEOUT once; rows >= M and the
columns of the warp that gave up stay unwritten; every other column is right;
the argmax workspace is left zero; and the next normal call is exact."""
import time

import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SENT = np.float32(-3.25)
RTOL, ATOL = 1e-4, 1e-6
K, N = 2048, 512          # 8 chunks of 256: three ring stages per warp unit
SHAPE = (16, 2, 1)        # one CTA per 16-column tile pair; CTA 0 owns columns 0..15


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


@pytest.fixture(scope="module")
def case():
    mat = synth.Matrix("waits", synth.SIGN1_G128, K, N, 128, "f16")
    parts, xb = synth.gen_matrix(mat, 11)
    Wp = torch.from_numpy(lbv.pack(lbv.FMT_SIGN1_G128, parts, K, N, 128)).cuda()
    X = torch.from_numpy(xb.view(np.int16)).cuda()
    Yref, A = oracle.verify(lbv.FMT_SIGN1_G128, parts, oracle.x_to_f64(xb, "f16"), K, N, 128)
    return Wp, X, Yref, RTOL * A + ATOL


def plan(flags):
    p = lbv.Plan(lbv.FMT_SIGN1_G128, K, N, 128, lbv.F16, flags)
    p.set_shape(*SHAPE)
    return p


def test_flag_combinations_rejected():
    for bad in (lbv.PLAN_MEASURE, lbv.PLAN_FORCE_GEMV, lbv.PLAN_TCGEN05):
        with pytest.raises(lbv.LbvError) as e:
            lbv.Plan(lbv.FMT_SIGN1_G128, K, N, 128, lbv.F16, lbv.PLAN_TEST_WAIT_LIMIT | bad)
        assert e.value.status == lbv.ERR_INVALID_ARG


@pytest.mark.parametrize("M", [3, 8])
def test_wait_runs_out_and_kernel_returns(case, M):
    Wp, X, Yref, tol = case
    P = plan(lbv.PLAN_TEST_WAIT_LIMIT)
    assert P.shape()[:3] == SHAPE and P.shape()[3] == N // 16
    Y = torch.full((8, N), float(SENT), dtype=torch.float32, device="cuda")
    t0 = time.perf_counter()
    lbv.verify_gemm(P, X, M, Wp, Y)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    with pytest.raises(lbv.LbvError) as e:
        P.device_status()
    assert e.value.status == lbv.ERR_TIMEOUT
    P.device_status()                                 # reported once, then cleared
    got = Y.cpu().numpy()
    assert np.all(got[M:] == SENT)                    # rows >= M untouched
    assert np.all(got[:M, :16] == SENT)               # the warp that gave up stored nothing
    err = np.abs(got[:M, 16:].astype(np.float64) - Yref[:M, 16:])
    assert np.all(err <= tol[:M, 16:])                # every other column is right
    # the context is fine and the next normal call, same launch shape, is exact
    Q = plan(0)
    Y2 = torch.full((8, N), float(SENT), dtype=torch.float32, device="cuda")
    lbv.verify_gemm(Q, X, M, Wp, Y2)
    torch.cuda.synchronize()
    Q.device_status()
    got2 = Y2.cpu().numpy()
    assert np.all(np.abs(got2[:M].astype(np.float64) - Yref[:M]) <= tol[:M])
    assert np.array_equal(got2[:M, 16:], got[:M, 16:])
    assert np.all(got2[M:] == SENT)


def test_wait_runs_out_in_argmax_head(case):
    """The fused argmax epilogue after a give-up: the call ends, the status
    reports the timeout, the workspace is left zero for the next call, and
    the next normal call gives the argmax of its own logits."""
    Wp, X, Yref, tol = case
    P = plan(lbv.PLAN_TEST_WAIT_LIMIT)
    ws = torch.zeros(lbv.fused_workspace_bytes(), dtype=torch.uint8, device="cuda")
    idx = torch.full((8,), -9, dtype=torch.int32, device="cuda")
    lbv.verify_fused(P, X, 8, Wp, lbv.FUSED_ARGMAX, idx=idx, workspace=ws)
    torch.cuda.synchronize()
    with pytest.raises(lbv.LbvError) as e:
        P.device_status()
    assert e.value.status == lbv.ERR_TIMEOUT
    assert np.all(ws.cpu().numpy() == 0)
    ig = idx.cpu().numpy()
    assert np.all((ig >= -1) & (ig < N))
    Q = plan(0)
    Y = torch.empty((8, N), dtype=torch.float32, device="cuda")
    lbv.verify_fused(Q, X, 8, Wp, lbv.FUSED_ARGMAX, Y=Y, idx=idx, workspace=ws)
    torch.cuda.synchronize()
    Q.device_status()
    Yg = Y.cpu().numpy()
    for m in range(8):
        assert idx.cpu().numpy()[m] == int(np.flatnonzero(Yg[m] == Yg[m].max())[0])
    assert np.all(ws.cpu().numpy() == 0)
