"""Leading dimensions and limits: X and Y with padded rows (ldx > K, ldy > N),
including X rows that are not 16-byte aligned (the element-wise staging
path), through the plain, fused and grouped calls; and a grouped call at the
256-problem limit.  Results are checked against the fp64 oracle and, where a
dense-row call exists, bit for bit against it."""
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
SENT = np.float32(-12345.5)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gen(fmtname, K, N, group, xdtype, seed):
    mat = synth.Matrix("s", fmtname, K, N, group, xdtype,
                       sigma_scale=0.02 if fmtname == synth.SIGN1_G128 else 0.01)
    return synth.gen_matrix(mat, seed, rows=8)


def padded_x(xb, ldx):
    """X rows at stride ldx (elements) in a device buffer, padding filled with
    a large value that must never be read."""
    M, K = xb.shape
    buf = np.full((M, ldx), np.float16(3e4).view(np.uint16), np.uint16)
    buf[:, :K] = xb
    return dev(buf.view(np.int16))


@pytest.mark.parametrize("fmtname,K,N,group,xdtype", [
    (synth.SIGN1_G128, 640, 200, 128, "f16"),
    (synth.AFFINE2, 768, 136, 64, "bf16"),
    (synth.Q4_0, 1024, 72, 32, "f16"),
])
@pytest.mark.parametrize("dx,dy", [(8, 0), (3, 5), (1, 16)])
@pytest.mark.parametrize("flags", [0, lbv.PLAN_FORCE_GEMV])
def test_verify_strided(fmtname, K, N, group, xdtype, dx, dy, flags):
    """Odd ldx puts rows >= 1 on 2-byte boundaries: the few-row kernel stages
    them element-wise and the 1-row path (PLAN_FORCE_GEMV) reads 2-byte
    elements, so neither makes a misaligned wider load."""
    parts, xb = gen(fmtname, K, N, group, xdtype, K + dx)
    fmt = FMT[fmtname]
    plan = lbv.Plan(fmt, K, N, group, DT[xdtype], flags)
    Wp = dev(lbv.pack(fmt, parts, K, N, group))
    ldx, ldy = K + dx, N + dy
    Xp = padded_x(xb, ldx)
    X = dev(xb.view(np.int16))
    Yref, A = oracle.verify(fmt, parts, oracle.x_to_f64(xb, xdtype), K, N, group)
    for M in (1, 5, 8):
        Yp = torch.full((8, ldy), float(SENT), dtype=torch.float32, device="cuda")
        Y = torch.full((8, N), float(SENT), dtype=torch.float32, device="cuda")
        lbv.verify_gemm(plan, Xp, M, Wp, Yp, ldx=ldx, ldy=ldy)
        lbv.verify_gemm(plan, X, M, Wp, Y)
        torch.cuda.synchronize()
        plan.device_status()
        got = Yp.cpu().numpy()
        assert np.array_equal(got[:M, :N], Y.cpu().numpy()[:M])
        assert np.all(got[:, N:] == SENT) and np.all(got[M:] == SENT)
        assert np.all(np.abs(got[:M, :N] - Yref[:M]) <= RTOL * A[:M] + ATOL)


@pytest.mark.parametrize("dx,dy", [(8, 3), (3, 0)])
def test_fused_strided(dx, dy):
    K, N = 1280, 400
    parts, xb = gen(synth.AFFINE2, K, N, 128, "f16", 77 + dx)
    plan = lbv.Plan(lbv.FMT_AFFINE2, K, N, 128, lbv.F16)
    Wp = dev(lbv.pack(lbv.FMT_AFFINE2, parts, K, N, 128))
    ldx, ldy = K + dx, N + dy
    Xp, X = padded_x(xb, ldx), dev(xb.view(np.int16))
    ws = torch.zeros(lbv.fused_workspace_bytes(), dtype=torch.uint8, device="cuda")
    ops = lbv.FUSED_ROTATE | lbv.FUSED_ARGMAX
    for M in (2, 8):
        Yp = torch.full((8, ldy), float(SENT), dtype=torch.float32, device="cuda")
        Y = torch.full((8, N), float(SENT), dtype=torch.float32, device="cuda")
        i1 = torch.full((8,), -5, dtype=torch.int32, device="cuda")
        i2 = torch.full((8,), -5, dtype=torch.int32, device="cuda")
        lbv.verify_fused(plan, Xp, M, Wp, ops, Y=Yp, idx=i1, workspace=ws, ldx=ldx, ldy=ldy)
        lbv.verify_fused(plan, X, M, Wp, ops, Y=Y, idx=i2, workspace=ws)
        torch.cuda.synchronize()
        plan.device_status()
        got = Yp.cpu().numpy()
        assert np.array_equal(got[:M, :N], Y.cpu().numpy()[:M])
        assert np.all(got[:, N:] == SENT) and np.all(got[M:] == SENT)
        assert np.array_equal(i1.cpu().numpy(), i2.cpu().numpy())
    assert np.all(ws.cpu().numpy() == 0)


def test_grouped_strided_and_256_problems():
    """256 Q4_0 problems (the limit), each with padded X and Y rows and its own
    row count, against the oracle; a sample of them against single calls."""
    n = 256
    rng = np.random.default_rng(123)
    shapes = [(int(rng.choice([128, 256, 512])), int(rng.choice([16, 32, 48]))) for _ in range(n)]
    G = lbv.Group(lbv.FMT_Q4_0, 32, lbv.F16, shapes)
    probs, host = [], []
    for i, (K, N) in enumerate(shapes):
        parts, xb = gen(synth.Q4_0, K, N, 32, "f16", [5, i])
        M = int(rng.integers(0, 9))
        ldx, ldy = K + int(rng.integers(0, 4)) * 3, N + int(rng.integers(0, 3))
        Wp = dev(lbv.pack(lbv.FMT_Q4_0, parts, K, N, 32))
        Xp = padded_x(xb, ldx)
        Y = torch.full((8, ldy), float(SENT), dtype=torch.float32, device="cuda")
        probs.append((Xp, M, Wp, Y, ldx, ldy))
        host.append((parts, xb, K, N, M))
    lbv.verify_grouped(G, probs)
    torch.cuda.synchronize()
    G.device_status()
    for i, ((Xp, M, Wp, Y, ldx, ldy), (parts, xb, K, N, _)) in enumerate(zip(probs, host)):
        got = Y.cpu().numpy()
        assert np.all(got[M:] == SENT) and np.all(got[:, N:] == SENT), i
        if M == 0:
            continue
        Yref, A = oracle.verify(lbv.FMT_Q4_0, parts, oracle.x_to_f64(xb[:M], "f16"), K, N, 32)
        assert np.all(np.abs(got[:M, :N] - Yref) <= RTOL * A + ATOL), i
        if i % 37 == 0:
            tpw, sp, _ = G.shape(G.problem_launch(i))
            plan = lbv.Plan(lbv.FMT_Q4_0, K, N, 32, lbv.F16)
            plan.set_shape(16, tpw, sp, 0)
            Y1 = torch.full((8, N), float(SENT), dtype=torch.float32, device="cuda")
            lbv.verify_gemm(plan, dev(xb.view(np.int16)), M, Wp, Y1)
            torch.cuda.synchronize()
            assert np.array_equal(got[:M, :N], Y1.cpu().numpy()[:M]), i
