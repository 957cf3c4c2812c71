"""GPU parity of the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerance (per output element, fp32 accumulation):
    |y_gpu - y_ref| <= 1e-4 * sum_k |x_k w_k| + 1e-6
with x the kernel's actual input (the rotated, rounded activations for the
rotated head) and w the exact weights.  Dequantized fp16 weights and the
FWHT-128 output are compared bit for bit.
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
SENTINEL = np.float32(-12345.5)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def x_dev(xb):
    return dev(xb.view(np.int16))


class Case:
    """Inputs of one matrix on host and device plus its oracle result."""

    def __init__(self, fmtname, K, N, group, xdtype, seed, cols=None, flags=0, rotate=False):
        self.mat = synth.Matrix("w", fmtname, K, N, group, xdtype, rotate=rotate,
                                sigma_scale=0.02 if fmtname == synth.SIGN1_G128 else 0.01)
        self.fmt = FMT[fmtname]
        self.K, self.N, self.group, self.xdtype = K, N, group, xdtype
        self.parts, self.xb = synth.gen_matrix(self.mat, seed, rows=8)
        self.plan = lbv.Plan(self.fmt, K, N, group, DT[xdtype], flags)
        # the layout this plan's kernels read (lbv_plan_pack)
        self.packed = lbv.pack(self.fmt, self.parts, K, N, group, plan=self.plan)
        self.Wp = dev(self.packed)
        self.X = x_dev(self.xb)
        self.cols = np.arange(N) if cols is None else np.asarray(cols)
        self.Xf = oracle.x_to_f64(self.xb, xdtype)
        self.Yref, self.A = oracle.verify(self.fmt, self.parts, self.Xf, K, N, group,
                                          cols=self.cols)

    def run(self, M, X=None, plan=None):
        Y = torch.full((8, self.N), float(SENTINEL), dtype=torch.float32, device="cuda")
        lbv.verify_gemm(plan or self.plan, self.X if X is None else X, M, self.Wp, Y)
        torch.cuda.synchronize()
        (plan or self.plan).device_status()
        return Y.cpu().numpy()

    def check(self, Y, M):
        got = Y[:M][:, self.cols].astype(np.float64)
        err = np.abs(got - self.Yref[:M])
        tol = RTOL * self.A[:M] + ATOL
        bad = err > tol
        assert not bad.any(), (f"{bad.sum()} of {bad.size} outside tolerance; worst "
                               f"{(err / tol).max():.3g}x tol at {np.argwhere(bad)[:5].tolist()}")
        assert np.all(Y[M:] == SENTINEL), "rows >= M were written"


SMALL = [
    # fmt, K, N, group, xdtype
    (synth.SIGN1_G128, 512, 256, 128, "f16"),    # the tiny 1-bit case
    (synth.SIGN1_G128, 1408, 200, 128, "f16"),   # ragged K chunk and N tail
    (synth.SIGN1_G128, 640, 96, 128, "bf16"),
    (synth.AFFINE2, 768, 136, 64, "bf16"),
    (synth.AFFINE2, 640, 40, 128, "f16"),
    (synth.AFFINE2, 352, 56, 32, "f16"),
    (synth.AFFINE2, 320, 24, 64, "f16"),
    (synth.AFFINE2, 384, 33, 128, "bf16"),
    (synth.Q4_0, 800, 72, 32, "f16"),
    (synth.Q4_0, 1024, 48, 32, "bf16"),
]


@pytest.mark.parametrize("fmtname,K,N,group,xdtype", SMALL)
def test_parity_small_all_M(fmtname, K, N, group, xdtype):
    c = Case(fmtname, K, N, group, xdtype, seed=0)
    for M in range(1, 9):
        c.check(c.run(M), M)


def test_tiny_1bit_seed0_every_shape():
    """The 512x256 1-bit case under every launch shape (warps, tiles per warp,
    K split): all within tolerance, each shape deterministic."""
    c = Case(synth.SIGN1_G128, 512, 256, 128, "f16", seed=0)
    seen = 0
    for warps, tpw in ((8, 2), (8, 4), (16, 1), (16, 2)):
        for splits in (1, 2):
            c.plan.set_shape(warps, tpw, splits)
            assert c.plan.shape()[:3] == (warps, tpw, splits)
            for M in (1, 5, 8):
                Y1, Y2 = c.run(M), c.run(M)
                assert np.array_equal(Y1, Y2)
                c.check(Y1, M)
            seen += 1
    assert seen == 8


@pytest.mark.parametrize("fmtname,K,N,group,xdtype", [
    (synth.SIGN1_G128, 2048, 160, 128, "f16"),
    (synth.AFFINE2, 1536, 96, 64, "bf16"),
    (synth.Q4_0, 1280, 80, 32, "f16")])
def test_split_k_shapes(fmtname, K, N, group, xdtype):
    c = Case(fmtname, K, N, group, xdtype, seed=3)
    tried = 0
    for splits in (1, 2, 3, 4, 5, 8):
        for ctas in (0, 1, 3):
            for warps, tpw in ((16, 1), (8, 4), (16, 2)):
                try:
                    c.plan.set_shape(warps, tpw, splits, ctas)
                except lbv.LbvError:
                    continue
                tried += 1
                for M in (2, 8):
                    c.check(c.run(M), M)
    assert tried >= 20


def test_row_and_M_independence_bitwise():
    """Row m of the result depends only on row m of X: an M-row call equals
    M single-row calls and the first rows of a larger call, bit for bit."""
    c = Case(synth.AFFINE2, 768, 112, 64, "bf16", seed=5)
    Y8 = c.run(8)
    for M in (1, 3, 7):
        assert np.array_equal(c.run(M)[:M], Y8[:M])
    for m in range(8):
        Ym = c.run(1, X=c.X[m:m + 1])
        assert np.array_equal(Ym[0], Y8[m])
    # changing another row's values changes nothing in row 0
    X2 = c.X.clone()
    X2[1:] = X2[1:].flip(0)
    Y = torch.zeros((8, c.N), dtype=torch.float32, device="cuda")
    lbv.verify_gemm(c.plan, X2, 8, c.Wp, Y)
    assert np.array_equal(Y.cpu().numpy()[0], Y8[0])


def test_gemv_path_parity_and_dispatch():
    for fmtname, K, N, group, xdtype in SMALL[:1] + SMALL[3:4] + SMALL[8:9]:
        c = Case(fmtname, K, N, group, xdtype, seed=2, flags=lbv.PLAN_FORCE_GEMV)
        for M in (1, 4):
            assert c.plan.query(M)[0] == lbv.KERNEL_GEMV
            c.check(c.run(M), M)
        c2 = Case(fmtname, K, N, group, xdtype, seed=2, flags=lbv.PLAN_FORCE_FEWROW)
        assert c2.plan.query(1)[0] == lbv.KERNEL_FEWROW


@pytest.mark.parametrize("K,N,xdtype", [
    (128, 16, "f16"), (384, 40, "bf16"), (1408, 200, "f16"), (5120, 72, "f16"),
    (5632, 24, "bf16"), (5888, 24, "f16")])
def test_gemv_sign1_table_path(K, N, xdtype):
    """The 1-bit 1-row path reads its codes through a per-CTA table of signed
    4-activation sums; K spans one chunk, ragged chunks, the largest K whose
    table and code buffers fit in shared memory (22 chunks) and the next one
    (the generic 1-row kernel).  Rows >= M stay untouched; repeated calls
    agree bitwise."""
    c = Case(synth.SIGN1_G128, K, N, 128, xdtype, seed=5, flags=lbv.PLAN_FORCE_GEMV)
    for M in (1, 3, 8):
        assert c.plan.query(M)[0] == lbv.KERNEL_GEMV
        Y = c.run(M)
        c.check(Y, M)
        assert np.array_equal(Y, c.run(M))


def test_pdl_back_to_back():
    """Programmatic dependent launch: a chain of calls where each call's X is
    the previous call's output (rounded to fp16 by a torch kernel in between)
    and calls that write Y right after the previous read it."""
    c = Case(synth.SIGN1_G128, 1024, 1024, 128, "f16", seed=4, flags=lbv.PLAN_PDL)
    plain = lbv.Plan(c.fmt, c.K, c.N, 128, lbv.F16, 0)
    Ys = []
    for plan in (c.plan, plain):
        X = c.X.clone()
        Y = torch.zeros((8, c.N), dtype=torch.float32, device="cuda")
        for _ in range(6):
            lbv.verify_gemm(plan, X, 8, c.Wp, Y)
            X = (Y[:, :c.K] * 0.05).half().view(torch.int16).contiguous()
        torch.cuda.synchronize()
        Ys.append(Y.cpu().numpy())
    assert np.array_equal(Ys[0], Ys[1])


@pytest.mark.parametrize("fmtname,K,N,group", [
    (synth.SIGN1_G128, 640, 40, 128), (synth.AFFINE2, 384, 56, 64), (synth.AFFINE2, 256, 24, 128),
    (synth.AFFINE2, 224, 17, 32), (synth.Q4_0, 352, 33, 32)])
def test_dequant_bit_exact(fmtname, K, N, group):
    mat = synth.Matrix("w", fmtname, K, N, group, "f16", sigma_scale=0.01)
    parts, _ = synth.gen_matrix(mat, 6, rows=1)
    fmt = FMT[fmtname]
    Wp = dev(lbv.pack(fmt, parts, K, N, group))
    plan = lbv.Plan(fmt, K, N, group, lbv.F16)
    W = torch.zeros((K, N), dtype=torch.int16, device="cuda")
    lbv.dequant_fp16(plan, Wp, W)
    torch.cuda.synchronize()
    got = W.cpu().numpy().view(np.uint16)
    ref = oracle.dequant_f16(fmt, parts, K, N, group)
    assert np.array_equal(got, ref)


def test_dequant_edge_values():
    """Scales at the fp16 extremes: subnormal, negative, zero, max."""
    K, N = 256, 16
    bits = np.random.default_rng(0).integers(0, 2**32, (N, K // 32), dtype=np.uint32)
    sc = np.array([0x0001, 0x03FF, 0x8001, 0x0000, 0x8000, 0x7BFF, 0xFBFF, 0x3C00] * 4,
                  np.uint16).reshape(N, K // 128)
    Wp = dev(lbv.pack_sign_g128(bits, sc, K, N))
    plan = lbv.Plan(lbv.FMT_SIGN1_G128, K, N, 128, lbv.F16)
    W = torch.zeros((K, N), dtype=torch.int16, device="cuda")
    lbv.dequant_fp16(plan, Wp, W)
    got = W.cpu().numpy().view(np.uint16)
    ref = oracle.dequant_f16(0, (bits, sc), K, N, 128)
    # +-0 are both exact zero weights; compare values, and bits where nonzero
    assert np.array_equal(got.view(np.float16).astype(np.float64), ref.view(np.float16).astype(np.float64))
    nz = ref.view(np.float16) != 0
    assert np.array_equal(got[nz], ref[nz])


@pytest.mark.parametrize("xdtype", ["f16", "bf16"])
@pytest.mark.parametrize("with_signs", [False, True])
def test_fwht128_bit_exact(xdtype, with_signs):
    rng = np.random.default_rng(7)
    M, K = 8, 5120
    xb = synth.x_bits(rng, M, K, xdtype)
    signs = synth.random_signs(8, K) if with_signs else None
    X = x_dev(xb)
    Xr = torch.zeros_like(X)
    lbv.fwht128(X, Xr, M, K, DT[xdtype], None if signs is None else dev(signs.view(np.int32)))
    torch.cuda.synchronize()
    got = Xr.cpu().numpy().view(np.uint16)
    ref = oracle.round_x(oracle.fwht128(oracle.x_to_f64(xb, xdtype), signs), xdtype)
    assert np.array_equal(got, ref)
    # in place
    lbv.fwht128(X, X, M, K, DT[xdtype], None if signs is None else dev(signs.view(np.int32)))
    torch.cuda.synchronize()
    assert np.array_equal(X.cpu().numpy().view(np.uint16), ref)


def test_rotated_head_small():
    """FWHT-128 then 2-bit affine g128 against the oracle on the rotated,
    rounded activations; and the rotation invariance of the exact product."""
    K, N = 1024, 200
    c = Case(synth.AFFINE2, K, N, 128, "f16", seed=9, rotate=True)
    Xr = torch.zeros_like(c.X)
    lbv.fwht128(c.X, Xr, 8, K, lbv.F16)
    xr_bits = oracle.round_x(oracle.fwht128(c.Xf), "f16")
    Yref, A = oracle.verify(c.fmt, c.parts, oracle.f16_to_f64(xr_bits), K, N, 128)
    for M in (1, 5, 8):
        Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
        lbv.verify_gemm(c.plan, Xr, M, c.Wp, Y)
        got = Y.cpu().numpy()[:M].astype(np.float64)
        assert np.all(np.abs(got - Yref[:M]) <= RTOL * A[:M] + ATOL)


def test_error_codes_on_device():
    c = Case(synth.Q4_0, 256, 32, 32, "f16", seed=1)
    Y = torch.zeros((8, 32), dtype=torch.float32, device="cuda")
    for M in (0, 9, -1):
        with pytest.raises(lbv.LbvError) as e:
            lbv.verify_gemm(c.plan, c.X, M, c.Wp, Y)
        assert e.value.status == lbv.ERR_INVALID_ARG
    with pytest.raises(lbv.LbvError):
        lbv.verify_gemm(c.plan, c.X, 2, c.Wp, Y, ldx=100)
    with pytest.raises(lbv.LbvError):
        lbv.verify_gemm(c.plan, c.X, 2, c.Wp.view(torch.uint8)[2:], Y)   # misaligned Wp
    with pytest.raises(lbv.LbvError) as e:
        c.plan.set_shape(3, 1, 1)
    assert e.value.status == lbv.ERR_INVALID_ARG
    assert c.plan.query(3)[2] == 0                # no workspace
