"""GPU parity of the grouped verify (lbv_verify_grouped): independent problems
of one format in one launch -- a Q4_0 layer stack, routed experts with their
own rows.  Each problem's result must equal, bit for bit, lbv_verify_gemm
with a plan of the same shape and K split, and lie within the verify
tolerance of the fp64 oracle; problems with M = 0 and rows >= M are never
written.
"""
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


class Problems:
    """Problems of one format: packed weights, X and Y on the device."""

    def __init__(self, fmtname, group, xdtype, shapes, seed, flags=0):
        self.fmtname, self.fmt, self.group, self.xdtype = fmtname, FMT[fmtname], group, xdtype
        self.shapes = list(shapes)
        self.mats, self.parts, self.xb, self.Wp, self.X = [], [], [], [], []
        for i, (K, N) in enumerate(self.shapes):
            mat = synth.Matrix(f"p{i}", fmtname, K, N, group, xdtype,
                               sigma_scale=0.02 if fmtname == synth.SIGN1_G128 else 0.01)
            parts, xb = synth.gen_matrix(mat, [seed, i], rows=8)
            self.mats.append(mat)
            self.parts.append(parts)
            self.xb.append(xb)
            self.Wp.append(dev(lbv.pack(self.fmt, parts, K, N, group)))
            self.X.append(dev(xb.view(np.int16)))
        self.G = lbv.Group(self.fmt, group, DT[xdtype], self.shapes, flags)

    def run(self, Ms):
        Ys = [torch.full((8, N), float(SENT), dtype=torch.float32, device="cuda")
              for _, N in self.shapes]
        lbv.verify_grouped(self.G, [(X, M, W, Y) for X, M, W, Y in
                                    zip(self.X, Ms, self.Wp, Ys)])
        torch.cuda.synchronize()
        self.G.device_status()
        return [Y.cpu().numpy() for Y in Ys]

    def single(self, i, M):
        """lbv_verify_gemm of problem i with its launch class's tiles per unit and K split."""
        K, N = self.shapes[i]
        tpw, splits, _ = self.G.shape(self.G.problem_launch(i))
        plan = lbv.Plan(self.fmt, K, N, self.group, DT[self.xdtype])
        plan.set_shape(16, tpw, splits, 0)
        Y = torch.full((8, N), float(SENT), dtype=torch.float32, device="cuda")
        lbv.verify_gemm(plan, self.X[i], M, self.Wp[i], Y)
        torch.cuda.synchronize()
        return Y.cpu().numpy()

    def check(self, Ys, Ms, singles=True):
        for i, (Y, M) in enumerate(zip(Ys, Ms)):
            K, N = self.shapes[i]
            assert np.all(Y[M:] == SENT), f"problem {i}: rows >= M={M} were written"
            if M == 0:
                continue
            if singles:
                assert np.array_equal(Y, self.single(i, M)), f"problem {i} differs from one call"
            Xf = oracle.x_to_f64(self.xb[i][:M], self.xdtype)
            Yref, A = oracle.verify(self.fmt, self.parts[i], Xf, K, N, self.group)
            err = np.abs(Y[:M].astype(np.float64) - Yref)
            tol = RTOL * A + ATOL
            assert np.all(err <= tol), f"problem {i}: worst {(err / tol).max():.3g}x tol"


LAYER = [(640, 96), (640, 32), (640, 32), (768, 80), (1280, 48), (1280, 40), (2048, 64)]


def test_q4_0_layer_like_group():
    P = Problems(synth.Q4_0, 32, "f16", LAYER, seed=1)
    for Ms in ([8] * 7, [1] * 7, [3, 8, 0, 5, 1, 8, 2]):
        P.check(P.run(Ms), Ms)


def test_two_launch_classes():
    """Problems whose X slice needs a K split next to one too short to be
    split (K = 128 is two Q4_0 chunks, one 128-element block): no split suits
    all, so two launch classes in one call, each problem equal to its single
    call."""
    shapes = [(17408, 64), (128, 96), (2048, 48), (17408, 32)]
    P = Problems(synth.Q4_0, 32, "f16", shapes, seed=8)
    assert P.G.launches() == 2
    assert P.G.problem_launch(0) == P.G.problem_launch(3) != P.G.problem_launch(1)
    assert P.G.shape(P.G.problem_launch(1))[1] == 1 and P.G.shape(P.G.problem_launch(0))[1] > 1
    with pytest.raises(lbv.LbvError):
        P.G.shape(2)
    for Ms in ([8, 8, 8, 8], [0, 3, 0, 1], [2, 0, 8, 0]):
        P.check(P.run(Ms), Ms)


def test_measured_shapes():
    """LBV_PLAN_MEASURE picks each class's split and rows by timing; results
    still equal single calls with the chosen split."""
    shapes = [(17408, 64), (128, 96), (2048, 48), (6144, 80)]
    P = Problems(synth.Q4_0, 32, "f16", shapes, seed=9, flags=lbv.PLAN_MEASURE | lbv.PLAN_PDL)
    assert P.G.launches() == 2
    Q = Problems(synth.Q4_0, 32, "f16", LAYER, seed=10, flags=lbv.PLAN_MEASURE)
    assert Q.G.launches() == 1
    Q.check(Q.run([8, 1, 0, 3, 8, 2, 5]), [8, 1, 0, 3, 8, 2, 5])
    for c in range(P.G.launches()):
        tpw, sp, rows = P.G.shape(c)
        assert tpw == 2 and 1 <= sp <= 8 and rows >= 1
    for Ms in ([8, 8, 8, 8], [1, 0, 5, 2]):
        P.check(P.run(Ms), Ms)


@pytest.mark.parametrize("fmtname,group,xdtype,shapes", [
    (synth.SIGN1_G128, 128, "f16", [(512, 256), (1408, 200), (640, 96), (2048, 16)]),
    (synth.AFFINE2, 64, "bf16", [(768, 136), (512, 64), (1536, 96)]),
    (synth.AFFINE2, 128, "f16", [(640, 40), (1280, 400)]),
    (synth.AFFINE2, 32, "f16", [(352, 56), (320, 24), (512, 48)]),
])
def test_formats(fmtname, group, xdtype, shapes):
    P = Problems(fmtname, group, xdtype, shapes, seed=2)
    rng = np.random.default_rng(3)
    for _ in range(2):
        Ms = [int(m) for m in rng.integers(0, 9, size=len(shapes))]
        Ms[0] = max(Ms[0], 1)
        P.check(P.run(Ms), Ms)


def test_routed_experts():
    """16 experts of one shape, each with the rows routed to it (0..8): one
    launch equals per-expert calls bit for bit, and a row's result does not
    depend on the other rows of its expert."""
    P = Problems(synth.AFFINE2, 64, "bf16", [(1024, 256)] * 16, seed=4)
    rng = np.random.default_rng(5)
    Ms = [int(m) for m in rng.integers(0, 9, size=16)]
    Ms[3], Ms[7] = 0, 8
    Ys = P.run(Ms)
    P.check(Ys, Ms)
    Ys8 = P.run([8] * 16)
    for i, M in enumerate(Ms):
        assert np.array_equal(Ys[i][:M], Ys8[i][:M])


def test_shapes_agree_bitwise():
    """The tile partition (cluster rows, tiles per unit) never changes a
    result; only the K split does, and every split stays within tolerance."""
    P = Problems(synth.Q4_0, 32, "bf16", LAYER, seed=6)
    Ms = [8, 2, 5, 8, 1, 8, 3]
    assert P.G.launches() == 1
    tpw0, s0, r0 = P.G.shape()
    base = P.run(Ms)
    P.check(base, Ms)
    tried = 0
    for tpw in (1, 2):
        for rows in (1, 7, 23, 200):
            try:
                P.G.set_shape(tpw, s0, rows)
            except lbv.LbvError:
                continue
            tried += 1
            Ys = P.run(Ms)
            for a, b in zip(Ys, base):
                assert np.array_equal(a, b)
    assert tried >= 5
    for s in (1, 2, 4, 5, 8):
        try:
            P.G.set_shape(2, s, 30)
        except lbv.LbvError:
            continue
        tried += 1
        P.check(P.run(Ms), Ms)
    assert tried >= 7


def test_all_skipped_and_errors():
    P = Problems(synth.Q4_0, 32, "f16", LAYER[:3], seed=7)
    Ys = P.run([0, 0, 0])
    assert all(np.all(Y == SENT) for Y in Ys)
    Y = torch.zeros((8, 96), dtype=torch.float32, device="cuda")
    with pytest.raises(lbv.LbvError) as e:
        lbv.verify_grouped(P.G, [(P.X[0], 9, P.Wp[0], Y), (None, 0, None, None),
                                 (None, 0, None, None)])
    assert e.value.status == lbv.ERR_INVALID_ARG
    with pytest.raises(lbv.LbvError) as e:
        lbv.verify_grouped(P.G, [(P.X[0], 1, None, Y), (None, 0, None, None),
                                 (None, 0, None, None)])
    assert e.value.status == lbv.ERR_INVALID_ARG
    with pytest.raises(lbv.LbvError) as e:
        lbv.verify_grouped(P.G, [(P.X[0], 1, P.Wp[0], Y, 600, 96), (None, 0, None, None),
                                 (None, 0, None, None)])
    assert e.value.status == lbv.ERR_INVALID_ARG                     # ldx < K
    with pytest.raises(lbv.LbvError) as e:
        P.G.set_shape(3, 1, 10)
    assert e.value.status == lbv.ERR_INVALID_ARG
    with pytest.raises(lbv.LbvError) as e:
        lbv.Group(lbv.FMT_Q4_0, 32, lbv.F16, [(96, 32), (100, 32)])
    assert e.value.status == lbv.ERR_INVALID_ARG
    with pytest.raises(lbv.LbvError) as e:
        lbv.Group(lbv.FMT_Q4_0, 32, lbv.F16, [(64, 32)] * 257)
    assert e.value.status == lbv.ERR_INVALID_ARG
