"""The largest K each format's few-row plan accepts.  A plan splits K across
up to 8 cluster CTAs so that each CTA's slice of X fits in shared memory beside
its weight ring; past the largest K where some split fits, plan creation must
return LBV_ERR_UNSUPPORTED rather than build a plan that overruns shared memory.
When K is a multiple of 128 the slices are whole 128-element blocks (so that the
fused rotation can run on them); otherwise they are whole chunks only, and a
format with chunks under 128 elements (Q4_0) reaches a little further.  So the
limit is searched in each of those two families of K.  At each limit the verify
must agree with the oracle at M = 1 and 8, on every column of a ragged N, with
rows >= M untouched."""
import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FMT = {synth.SIGN1_G128: lbv.FMT_SIGN1_G128, synth.AFFINE2: lbv.FMT_AFFINE2,
       synth.Q4_0: lbv.FMT_Q4_0}
DT = {"f16": lbv.F16, "bf16": lbv.BF16}
RTOL, ATOL = 1e-4, 1e-6
SENTINEL = np.float32(-12345.5)
N = 40                     # two full 16-column tiles and a ragged one
K_CAP = 1 << 20            # the search stops here: no format reaches it


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


def accepts(fmt, K, group, dt):
    try:
        p = lbv.Plan(fmt, K, N, group, dt, lbv.PLAN_PDL)
    except lbv.LbvError as e:
        assert e.status == lbv.ERR_UNSUPPORTED, (K, str(e))
        return False
    p.close()
    return True


def largest_k(fmt, group, dt, kof):
    """Largest accepted kof(j) over j >= 0, where acceptance is monotone in j
    within one family of K (the checks after the search confirm it near the
    edge)."""
    assert accepts(fmt, kof(1), group, dt)
    lo = 1
    while kof(lo * 2) <= K_CAP and accepts(fmt, kof(lo * 2), group, dt):
        lo *= 2
    assert kof(lo * 2) <= K_CAP, "no K limit found below the search cap"
    hi = lo * 2                                          # rejected
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if accepts(fmt, kof(mid), group, dt):
            lo = mid
        else:
            hi = mid
    return lo


@pytest.mark.parametrize("fmtname,group,xdtype,quantum", [
    (synth.SIGN1_G128, 128, "f16", 128), (synth.AFFINE2, 32, "f16", 32),
    (synth.AFFINE2, 64, "bf16", 64), (synth.AFFINE2, 128, "f16", 128),
    (synth.Q4_0, 32, "f16", 32)])
def test_largest_k(fmtname, group, xdtype, quantum):
    fmt, dt = FMT[fmtname], DT[xdtype]
    families = [lambda j: 128 * j]                       # whole 128-element slices
    if quantum < 128:
        families.append(lambda j: 128 * j + quantum)     # K not a multiple of 128
    limits = []
    for kof in families:
        j = largest_k(fmt, group, dt, kof)
        for dj in (1, 2, 8):
            assert not accepts(fmt, kof(j + dj), group, dt), kof(j + dj)
        limits.append(kof(j))
    assert min(limits) >= 17408                          # the widest matrix of the workloads
    print(f"largest K, {fmtname} g{group} {xdtype}: {limits}")

    for K in limits:
        mat = synth.Matrix("w", fmtname, K, N, group, xdtype,
                           sigma_scale=0.02 if fmtname == synth.SIGN1_G128 else 0.01)
        parts, xb = synth.gen_matrix(mat, 7, rows=8)
        plan = lbv.Plan(fmt, K, N, group, dt, lbv.PLAN_PDL)
        Wp = torch.from_numpy(lbv.pack(fmt, parts, K, N, group, plan=plan)).cuda()
        X = torch.from_numpy(xb.view(np.int16)).cuda()
        Yref, A = oracle.verify(fmt, parts, oracle.x_to_f64(xb, xdtype), K, N, group)
        for M in (1, 8):
            Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
            lbv.verify_gemm(plan, X, M, Wp, Y)
            torch.cuda.synchronize()
            plan.device_status()
            got = Y.cpu().numpy()
            err = np.abs(got[:M].astype(np.float64) - Yref[:M])
            tol = RTOL * A[:M] + ATOL
            assert np.all(err <= tol), f"K={K} M={M}: worst {(err / tol).max():.3g}x tol"
            assert np.all(got[M:] == SENTINEL)
        plan.close()
