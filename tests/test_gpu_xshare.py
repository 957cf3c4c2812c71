"""GPU tests of X-sharing pairs (LBV_PLAN_X_SHARE): without a K split, two CTAs
of a cluster along N each stage, rotate (fused head) and correct half of the K
range and copy their half into the other's shared memory.  The results must
equal those of unpaired CTAs (the default) bit for bit, and the oracle within
the verify tolerance, for every format, both activation dtypes, X that is not
16-byte aligned, and the fused rotation and argmax."""
import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import oracle
import synth
import test_gpu_fused as F
from test_gpu_parity import SENTINEL, Case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
XS = lbv.PLAN_X_SHARE
DT = {"f16": lbv.F16, "bf16": lbv.BF16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


CASES = [
    # fmt, K, N, group, xdtype, launch shape (warps, tpw) with no K split
    (synth.SIGN1_G128, 2048, 1000, 128, "f16", (16, 1)),
    (synth.SIGN1_G128, 1280, 520, 128, "bf16", (16, 2)),
    (synth.AFFINE2, 1536, 700, 64, "bf16", (16, 1)),
    (synth.AFFINE2, 1280, 2000, 128, "f16", (16, 2)),
    (synth.AFFINE2, 640, 300, 32, "f16", (8, 2)),
    (synth.Q4_0, 1024, 600, 32, "f16", (16, 2)),
    (synth.Q4_0, 800, 260, 32, "bf16", (8, 4)),     # K not a multiple of 128
]


@pytest.mark.parametrize("fmtname,K,N,group,xdtype,wt", CASES)
def test_xshare_equals_unpaired(fmtname, K, N, group, xdtype, wt):
    c = Case(fmtname, K, N, group, xdtype, seed=K + N, flags=XS)
    plain = lbv.Plan(c.fmt, K, N, group, DT[xdtype], 0)
    for ctas in (0, 16, 7):                 # 7: odd, so no pairs even with the flag
        c.plan.set_shape(*wt, 1, ctas)
        plain.set_shape(*wt, 1, ctas)
        assert c.plan.shape()[:3] == (*wt, 1)
        for M in (1, 5, 8):
            Y = c.run(M)
            c.check(Y, M)
            assert np.array_equal(Y, c.run(M, plan=plain)), f"ctas={ctas} M={M}"


@pytest.mark.parametrize("dx", [1, 8])
def test_xshare_strided_x(dx):
    """Row stride K + dx, and X one element into its buffer for odd dx (the
    plain-load staging path)."""
    K, N = 1024, 640
    c = Case(synth.AFFINE2, K, N, 64, "bf16", seed=3, flags=XS)
    plain = lbv.Plan(c.fmt, K, N, 64, lbv.BF16, 0)
    c.plan.set_shape(16, 1, 1, 0)
    plain.set_shape(16, 1, 1, 0)
    base = torch.zeros((8 * (K + dx) + 8,), dtype=torch.int16, device="cuda")
    off = 1 if dx % 2 else 0
    Xs = base[off:off + 8 * (K + dx)].view(8, K + dx)
    Xs[:, :K] = c.X
    for M in (2, 8):
        outs = []
        for plan in (c.plan, plain):
            Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
            lbv.verify_gemm(plan, Xs, M, c.Wp, Y, ldx=K + dx)
            torch.cuda.synchronize()
            plan.device_status()
            outs.append(Y.cpu().numpy())
        c.check(outs[0], M)
        assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("fmtname,K,N,group,xdtype,signs", [
    (synth.AFFINE2, 1280, 2000, 128, "f16", True),      # the head's format
    (synth.AFFINE2, 5120, 4096, 128, "f16", False),     # the head's K
    (synth.SIGN1_G128, 1024, 600, 128, "bf16", True),
    (synth.Q4_0, 1024, 600, 32, "f16", True)])
def test_xshare_fused_head(fmtname, K, N, group, xdtype, signs):
    """Fused rotation and argmax with each CTA of a pair rotating its half:
    logits bitwise equal to unpaired CTAs and to the exported rotation's
    verify, within tolerance of the oracle; the argmax valid."""
    c = F.Case(fmtname, K, N, group, xdtype, seed=K, flags=XS, signs=signs)
    d = F.Case(fmtname, K, N, group, xdtype, seed=K, flags=0, signs=signs)
    for case in (c, d):
        case.plan.set_shape(16, 2, 1, 0)
    Yref, A = c.oracle_y(rotate=True)
    Xr = c.exported_x()
    for M in (1, 8):
        Y, idx, val = c.fused(M, F.ROT | F.AMAX)
        Y2, idx2, val2 = d.fused(M, F.ROT | F.AMAX)
        assert np.array_equal(Y, Y2) and np.array_equal(idx, idx2)
        assert np.array_equal(Y, c.verify(M, Xr))
        assert np.all(np.abs(Y[:M] - Yref[:M]) <= F.RTOL * A[:M] + F.ATOL)
        F.check_argmax(Y, idx, val, M, Yref, A, N)
    assert np.all(c.ws.cpu().numpy() == 0)
