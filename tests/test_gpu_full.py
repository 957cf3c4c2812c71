"""GPU parity at the full workload sizes, in the launch configurations the
benchmark times.

Plans and groups are created exactly as bench.py creates them
(LBV_PLAN_MEASURE | LBV_PLAN_PDL: the launch shape is the one the plan's
measurement picks on this GPU, and the kernel each row count dispatches to is
the plan's), and the shapes that measurement picked on GB300 are also set
explicitly, so the timed instantiations are the tested ones whatever a given
run measures.  Every output column is compared with the fp64 oracle (computed
once per matrix at M = 8 over all columns on every host core; row m of an
M-row call must match row m of it, as the oracle's rows are independent),
within |y - y_ref| <= 1e-4 * sum_k |x_k w_k| + 1e-6.  Rows >= M stay untouched.
"""
import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import oracle
import synth
from oracle_cols import verify_all

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FMT = {synth.SIGN1_G128: lbv.FMT_SIGN1_G128, synth.AFFINE2: lbv.FMT_AFFINE2,
       synth.Q4_0: lbv.FMT_Q4_0}
DT = {"f16": lbv.F16, "bf16": lbv.BF16}
RTOL, ATOL = 1e-4, 1e-6
SENT = np.float32(-7.0)
BENCH_FLAGS = lbv.PLAN_MEASURE | lbv.PLAN_PDL

# Launch shapes (warps, tiles per warp unit, K split) that the plan
# measurement picked for the benchmark on GB300.
GB300_SHAPES = {
    "sign1_mlp_up_5120x17408": [(16, 1, 1), (8, 2, 1)],
    "affine2_g64_6144x6144": [(16, 1, 4), (8, 2, 4)],
    "affine2_g64_kv_5120x1024": [(8, 2, 7), (8, 2, 8)],
    "head_rot_affine2_g128_5120x151936": [(16, 2, 1)],
}
# Grouped launch shapes (tiles per unit, K split, cluster rows) of the Q4_0 stack.
GB300_STACK_SHAPES = [(2, 4, 180), (2, 4, 144)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def reference(mat, parts, xb, rotate=False):
    """Oracle Y and tolerance scale A for all 8 rows and all columns."""
    Xf = oracle.x_to_f64(xb, mat.xdtype)
    if rotate:
        Xf = oracle.x_to_f64(oracle.round_x(oracle.fwht128(Xf), mat.xdtype), mat.xdtype)
    return verify_all(FMT[mat.fmt], parts, Xf, mat.K, mat.N, mat.group)


def check(got, M, Yref, A, what):
    err = np.abs(got[:M].astype(np.float64) - Yref[:M])
    tol = RTOL * A[:M] + ATOL
    assert np.all(err <= tol), f"{what} M={M}: worst {(err / tol).max():.3g}x tol"
    assert np.all(got[M:] == SENT), f"{what} M={M}: rows >= M written"


class Single:
    """One matrix of a workload on the device, with a plan made as the bench makes it."""

    def __init__(self, mat, parts, xb, rotate=False):
        self.mat = mat
        self.fmt = FMT[mat.fmt]
        self.plan = lbv.Plan(self.fmt, mat.K, mat.N, mat.group, DT[mat.xdtype], BENCH_FLAGS)
        self.Wp = dev(lbv.pack(self.fmt, parts, mat.K, mat.N, mat.group, plan=self.plan))
        self.X = dev(xb.view(np.int16))
        self.rotate = rotate

    def run(self, M):
        Y = torch.full((8, self.mat.N), float(SENT), dtype=torch.float32, device="cuda")
        if self.rotate:
            lbv.verify_fused(self.plan, self.X, M, self.Wp, lbv.FUSED_ROTATE, Y=Y)
        else:
            lbv.verify_gemm(self.plan, self.X, M, self.Wp, Y)
        torch.cuda.synchronize()
        self.plan.device_status()       # no bounded wait gave up
        return Y.cpu().numpy()


def check_single(name, rotate=False):
    (mat, parts, xb), = synth.gen_workload(name)
    Yref, A = reference(mat, parts, xb, rotate)
    s = Single(mat, parts, xb, rotate)
    measured = s.plan.shape()
    for M in range(1, 9):
        kernel, splits, _ = s.plan.query(M)
        assert kernel in (lbv.KERNEL_FEWROW, lbv.KERNEL_GEMV)
        if kernel == lbv.KERNEL_FEWROW:
            assert splits == measured[2]
        check(s.run(M), M, Yref, A, f"{name} measured shape {measured}")
    for warps, tpw, splits in GB300_SHAPES.get(name, []):
        s.plan.set_shape(warps, tpw, splits)
        assert s.plan.shape()[:3] == (warps, tpw, splits)
        for M in (1, 5, 8):
            Y = s.run(M) if s.plan.query(M)[0] == lbv.KERNEL_FEWROW else None
            if Y is not None:
                check(Y, M, Yref, A, f"{name} shape {(warps, tpw, splits)}")
        # both calls of one shape agree bit for bit
        if s.plan.query(8)[0] == lbv.KERNEL_FEWROW:
            assert np.array_equal(s.run(8), s.run(8))
    return s, Yref, A


@pytest.mark.parametrize("name", ["sign1_tiny_512x256", "sign1_mlp_up_5120x17408",
                                  "affine2_g64_6144x6144", "affine2_g64_kv_5120x1024"])
def test_full_config(name):
    check_single(name)


def test_full_rotated_head():
    """The rotated output head as the bench runs it: FWHT-128 fused into the
    verify prologue, every one of the 151936 columns."""
    check_single("head_rot_affine2_g128_5120x151936", rotate=True)


def test_full_head_greedy_argmax():
    """The greedy head (fused rotation and per-row argmax, no logits): the
    chosen column is the first maximum of the same launch shape's logits and a
    valid choice against the oracle over all columns."""
    (mat, parts, xb), = synth.gen_workload("head_rot_affine2_g128_5120x151936")
    Yref, A = reference(mat, parts, xb, rotate=True)
    s = Single(mat, parts, xb, rotate=True)
    ws = torch.zeros(lbv.fused_workspace_bytes(), dtype=torch.uint8, device="cuda")
    for M in (1, 8):
        idx = torch.full((8,), -5, dtype=torch.int32, device="cuda")
        val = torch.zeros(8, dtype=torch.float32, device="cuda")
        lbv.verify_fused(s.plan, s.X, M, s.Wp, lbv.FUSED_ROTATE | lbv.FUSED_ARGMAX,
                         idx=idx, val=val, workspace=ws)
        Y = s.run(M)
        s.plan.device_status()
        ig, vg = idx.cpu().numpy(), val.cpu().numpy()
        assert np.all(ig[M:] == -5)
        tol = RTOL * A + ATOL
        for m in range(M):
            first = int(np.flatnonzero(Y[m] == Y[m].max())[0])
            assert ig[m] == first and vg[m] == Y[m, first]
            best = int(np.argmax(Yref[m]))
            assert Yref[m, ig[m]] >= Yref[m, best] - tol[m, ig[m]] - tol[m, best]
    assert np.all(ws.cpu().numpy() == 0)


@pytest.fixture(scope="module")
def stack():
    gen = list(synth.gen_workload("q4_0_stack_4x7"))
    refs = [reference(m, parts, xb) for m, parts, xb in gen]
    Wp = [dev(lbv.pack(lbv.FMT_Q4_0, parts, m.K, m.N, 32)) for m, parts, _ in gen]
    X = [dev(xb.view(np.int16)) for _, _, xb in gen]
    return gen, refs, Wp, X


def run_group(G, stack, M):
    gen, _, Wp, X = stack
    Ys = [torch.full((8, m.N), float(SENT), dtype=torch.float32, device="cuda")
          for m, _, _ in gen]
    lbv.verify_grouped(G, [(x, M, w, y) for x, w, y in zip(X, Wp, Ys)])
    torch.cuda.synchronize()
    G.device_status()
    return [Y.cpu().numpy() for Y in Ys]


def test_full_q4_0_stack_grouped(stack):
    """The 4 x 7 Q4_0 stack in one grouped launch, as the bench runs it
    (measured group shape, PDL) and with the group shapes measured on GB300;
    every column of all 28 matrices."""
    gen, refs, _, _ = stack
    shapes = [(m.K, m.N) for m, _, _ in gen]
    G = lbv.Group(lbv.FMT_Q4_0, 32, lbv.F16, shapes, BENCH_FLAGS)
    measured = [G.shape(c) for c in range(G.launches())]
    for M in (1, 3, 8):
        for (m, _, _), Y, (Yref, A) in zip(gen, run_group(G, stack, M), refs):
            check(Y, M, Yref, A, f"{m.name} grouped {measured}")
    for tpw, splits, rows in GB300_STACK_SHAPES:
        G.set_shape(tpw, splits, rows)
        assert G.shape(0) == (tpw, splits, rows)
        for M in (1, 8):
            for (m, _, _), Y, (Yref, A) in zip(gen, run_group(G, stack, M), refs):
                check(Y, M, Yref, A, f"{m.name} grouped {(tpw, splits, rows)}")


def test_full_q4_0_stack_calls(stack):
    """The Q4_0 stack as one verify call per matrix (the bench's per-call
    rows): plans made as the bench makes them, every column."""
    gen, refs, Wp, X = stack
    plans = {}
    for (m, _, _), w, x, (Yref, A) in zip(gen, Wp, X, refs):
        key = (m.K, m.N)
        if key not in plans:
            plans[key] = lbv.Plan(lbv.FMT_Q4_0, m.K, m.N, 32, lbv.F16, BENCH_FLAGS)
        plan = plans[key]
        for M in (1, 8):
            Y = torch.full((8, m.N), float(SENT), dtype=torch.float32, device="cuda")
            lbv.verify_gemm(plan, x, M, w, Y)
            torch.cuda.synchronize()
            plan.device_status()
            check(Y.cpu().numpy(), M, Yref, A, f"{m.name} shape {plan.shape()}")
