"""GPU parity of the fused head (lbv_verify_fused): the blockwise FWHT-128
rotation as the verify kernel's prologue and the per-row greedy argmax as its
epilogue, through the C ABI, against the fp64 oracle.

What is compared:
  - the fused rotation (test export lbv_fused_rotation, the same device code)
    element by element with the exact rotation: within one unit in the last
    place plus the fp32 sum error bound 2^-20 * |x_b|_1 / sqrt(128) of the block,
    and bit-identical to the correctly rounded value in all but a few
    elements;
  - fused logits bit for bit against lbv_verify_gemm on the exported X', and
    within the verify tolerance of the oracle;
  - the argmax: the first maximum of the call's own fp32 logits (unique), and
    a valid choice for the exact logits: Y[idx] >= max Y - tol[idx] - tol[best].
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
SENT_Y = np.float32(-12345.5)
SENT_I = -77
ROT, AMAX = lbv.FUSED_ROTATE, lbv.FUSED_ARGMAX


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def workspace():
    return torch.zeros(lbv.fused_workspace_bytes(), dtype=torch.uint8, device="cuda")


def first_argmax(Y):
    """First maximum of each fp32 row (the kernel's own logits)."""
    return np.array([int(np.argmax(r)) for r in Y])


class Case:
    def __init__(self, fmtname, K, N, group, xdtype, seed, flags=0, signs=False, parts=None,
                 xb=None):
        mat = synth.Matrix("w", fmtname, K, N, group, xdtype,
                           sigma_scale=0.02 if fmtname == synth.SIGN1_G128 else 0.01)
        self.K, self.N, self.group, self.xdtype = K, N, group, xdtype
        self.fmt = FMT[fmtname]
        gp, gx = synth.gen_matrix(mat, seed, rows=8)
        self.parts = gp if parts is None else parts
        self.xb = gx if xb is None else xb
        self.plan = lbv.Plan(self.fmt, K, N, group, DT[xdtype], flags)
        self.Wp = dev(lbv.pack(self.fmt, self.parts, K, N, group, plan=self.plan))
        self.X = dev(self.xb.view(np.int16))
        self.signs_h = synth.random_signs(seed + 100, K) if signs else None
        self.signs = dev(self.signs_h.view(np.int32)) if signs else None
        self.ws = workspace()

    def oracle_x(self, rotate):
        Xf = oracle.x_to_f64(self.xb, self.xdtype)
        if rotate:
            Xf = oracle.x_to_f64(oracle.round_x(oracle.fwht128(Xf, self.signs_h), self.xdtype),
                                 self.xdtype)
        return Xf

    def oracle_y(self, rotate, cols=None):
        return oracle.verify(self.fmt, self.parts, self.oracle_x(rotate), self.K, self.N,
                             self.group, cols=cols)

    def fused(self, M, ops, want_y=True, want_val=True):
        Y = torch.full((8, self.N), float(SENT_Y), dtype=torch.float32, device="cuda") \
            if want_y else None
        idx = torch.full((8,), SENT_I, dtype=torch.int32, device="cuda")
        val = torch.full((8,), float(SENT_Y), dtype=torch.float32, device="cuda")
        lbv.verify_fused(self.plan, self.X, M, self.Wp, ops, Y=Y, idx=idx,
                         val=val if want_val else None, workspace=self.ws,
                         signs=self.signs if ops & ROT else None)
        torch.cuda.synchronize()
        self.plan.device_status()
        return (None if Y is None else Y.cpu().numpy(), idx.cpu().numpy(), val.cpu().numpy())

    def exported_x(self):
        Xr = torch.zeros_like(self.X)
        lbv.fused_rotation(self.X, Xr, 8, self.K, DT[self.xdtype], signs=self.signs)
        torch.cuda.synchronize()
        return Xr

    def verify(self, M, X):
        Y = torch.full((8, self.N), float(SENT_Y), dtype=torch.float32, device="cuda")
        lbv.verify_gemm(self.plan, X, M, self.Wp, Y)
        torch.cuda.synchronize()
        return Y.cpu().numpy()


def check_argmax(Y, idx, val, M, Yref, A, N):
    """idx/val against the call's own logits (exactly) and the oracle (validity)."""
    assert np.all(idx[M:] == SENT_I), "rows >= M of the argmax were written"
    assert np.all(val[M:] == SENT_Y)
    if Y is not None:
        assert np.array_equal(idx[:M], first_argmax(Y[:M, :N]))
        assert np.array_equal(val[:M].view(np.uint32),
                              Y[np.arange(M), idx[:M]].view(np.uint32))
    tol = RTOL * A[:M] + ATOL
    best = oracle.argmax_rows(Yref[:M])
    r = np.arange(M)
    ok = Yref[r, idx[:M]] >= Yref[r, best] - tol[r, idx[:M]] - tol[r, best]
    assert ok.all(), f"argmax not a valid greedy choice in rows {np.flatnonzero(~ok).tolist()}"


def ulp_up(bits, xdtype):
    """Gap from |v| to the next larger representable magnitude."""
    mag = bits & 0x7FFF
    a = oracle.x_to_f64(mag.astype(np.uint16), xdtype)
    b = oracle.x_to_f64((mag + 1).astype(np.uint16), xdtype)
    return b - a


# ----------------------------------------------------------------------------
# the rotation itself

@pytest.mark.parametrize("xdtype,K,signs", [("f16", 1024, False), ("f16", 640, True),
                                            ("bf16", 1152, False), ("bf16", 256, True)])
def test_fused_rotation_elementwise(xdtype, K, signs):
    rng = np.random.default_rng(K)
    xb = synth.x_bits(rng, 8, K, xdtype)
    sg = synth.random_signs(K + 1, K) if signs else None
    X = dev(xb.view(np.int16))
    for M in (8, 3):
        Xr = torch.full_like(X, 0x5555)
        lbv.fused_rotation(X, Xr, M, K, DT[xdtype],
                           signs=dev(sg.view(np.int32)) if signs else None)
        torch.cuda.synchronize()
        got = Xr.cpu().numpy().view(np.uint16)
        assert np.all(got[M:] == 0x5555), "rows >= M were written"
        xf = oracle.x_to_f64(xb[:M], xdtype)
        exact = oracle.fwht128(xf, sg)                       # fp64, unrounded
        rne = oracle.round_x(exact, xdtype)
        q = oracle.x_to_f64(got[:M], xdtype)
        l1 = np.abs(xf).reshape(M, K // 128, 128).sum(-1) / np.sqrt(128.0)
        slack = np.repeat(2.0 ** -20 * l1, 128, axis=1)
        bound = ulp_up(rne, xdtype) + slack
        assert np.all(np.abs(q - exact) <= bound), \
            f"worst {(np.abs(q - exact) / bound).max():.3g}x bound"
        mismatch = np.mean(got[:M] != rne)
        assert mismatch < 0.01, f"{mismatch:.4f} of elements differ from the rounded rotation"


def test_fused_rotation_in_place_and_closed_form():
    """e_j * v rotates to v/sqrt(128) * H row j (closed form, exact after
    rounding for v = sqrt(128)); in place gives the same as out of place."""
    K = 256
    xb = np.zeros((8, K), np.uint16)
    v = np.float16(np.sqrt(128.0))
    for m in range(8):
        xb[m, 37 * m % K] = v.view(np.uint16)
    X = dev(xb.view(np.int16))
    Xr = torch.zeros_like(X)
    lbv.fused_rotation(X, Xr, 8, K, lbv.F16)
    lbv.fused_rotation(X, X, 8, K, lbv.F16)
    torch.cuda.synchronize()
    a, b = Xr.cpu().numpy().view(np.uint16), X.cpu().numpy().view(np.uint16)
    assert np.array_equal(a, b)
    scale = float(v) / np.sqrt(128.0)
    for m in range(8):
        j = 37 * m % K
        blk = j // 128
        want = np.zeros(K)
        i = np.arange(128)
        want[blk * 128:(blk + 1) * 128] = scale * (-1.0) ** np.array(
            [bin(ii & (j % 128)).count("1") for ii in i])
        assert np.array_equal(a[m], oracle.round_x(want, "f16"))


# ----------------------------------------------------------------------------
# fused logits

@pytest.mark.parametrize("fmtname,K,N,group,xdtype,signs", [
    (synth.AFFINE2, 1280, 400, 128, "f16", False),     # the head's format
    (synth.AFFINE2, 1280, 400, 128, "f16", True),
    (synth.AFFINE2, 768, 136, 64, "bf16", True),
    (synth.SIGN1_G128, 1024, 200, 128, "f16", False),
    (synth.Q4_0, 1024, 96, 32, "bf16", False),
])
def test_fused_rotate_logits(fmtname, K, N, group, xdtype, signs):
    c = Case(fmtname, K, N, group, xdtype, seed=K + N, signs=signs)
    Yref, A = c.oracle_y(rotate=True)
    Xr = c.exported_x()
    for M in range(1, 9):
        Y, idx, val = c.fused(M, ROT)
        assert np.all(idx == SENT_I) and np.all(val == SENT_Y), "argmax written without the op"
        # bit for bit the plain verify of the exported rotation
        assert np.array_equal(Y, c.verify(M, Xr))
        err = np.abs(Y[:M].astype(np.float64) - Yref[:M])
        tol = RTOL * A[:M] + ATOL
        assert np.all(err <= tol), f"M={M}: worst {(err / tol).max():.3g}x tol"
        assert np.all(Y[M:] == SENT_Y)


def test_fused_rotate_split_shapes():
    """K split across cluster CTAs: each CTA rotates its own slice."""
    c = Case(synth.AFFINE2, 2048, 160, 128, "f16", seed=9, signs=True)
    Yref, A = c.oracle_y(rotate=True)
    Xr = c.exported_x()
    tried = 0
    for splits in (2, 4, 8):
        for warps, tpw in ((16, 1), (8, 2)):
            try:
                c.plan.set_shape(warps, tpw, splits)
            except lbv.LbvError:
                continue
            tried += 1
            for M in (1, 8):
                Y, idx, val = c.fused(M, ROT | AMAX)
                assert np.array_equal(Y, c.verify(M, Xr))
                assert np.all(np.abs(Y[:M] - Yref[:M]) <= RTOL * A[:M] + ATOL)
                check_argmax(Y, idx, val, M, Yref, A, c.N)
    assert tried >= 3


# ----------------------------------------------------------------------------
# argmax epilogue

SMALL = [
    (synth.SIGN1_G128, 512, 256, 128, "f16"),
    (synth.SIGN1_G128, 1408, 200, 128, "bf16"),
    (synth.AFFINE2, 768, 136, 64, "bf16"),
    (synth.AFFINE2, 352, 56, 32, "f16"),
    (synth.AFFINE2, 640, 2000, 128, "f16"),
    (synth.Q4_0, 800, 72, 32, "f16"),
    (synth.Q4_0, 1024, 1040, 32, "bf16"),
]


@pytest.mark.parametrize("fmtname,K,N,group,xdtype", SMALL)
def test_argmax_all_M(fmtname, K, N, group, xdtype):
    c = Case(fmtname, K, N, group, xdtype, seed=N)
    Yref, A = c.oracle_y(rotate=False)
    for M in range(1, 9):
        Y, idx, val = c.fused(M, AMAX)
        assert np.array_equal(Y, c.verify(M, c.X)), "logits differ from lbv_verify_gemm"
        check_argmax(Y, idx, val, M, Yref, A, N)
        # argmax only: no logits written, the same choice and value
        _, idx2, val2 = c.fused(M, AMAX, want_y=False)
        assert np.array_equal(idx2, idx) and np.array_equal(val2.view(np.uint32),
                                                            val.view(np.uint32))
        _, idx3, val3 = c.fused(M, AMAX, want_y=False, want_val=False)
        assert np.array_equal(idx3, idx) and np.all(val3 == SENT_Y)
    assert np.all(c.ws.cpu().numpy() == 0), "workspace not left zeroed"


def test_argmax_every_shape():
    c = Case(synth.AFFINE2, 1536, 1000, 64, "bf16", seed=4)
    Yref, A = c.oracle_y(rotate=False)
    tried = 0
    for warps, tpw in ((8, 2), (8, 4), (16, 1), (16, 2)):
        for splits in (1, 2, 3, 6):
            for ctas in (0, 1, 5):
                try:
                    c.plan.set_shape(warps, tpw, splits, ctas)
                except lbv.LbvError:
                    continue
                tried += 1
                for M in (1, 8):
                    Y, idx, val = c.fused(M, AMAX)
                    check_argmax(Y, idx, val, M, Yref, A, c.N)
    assert tried >= 20


@pytest.mark.parametrize("shape", [None, (16, 1, 2), (8, 4, 3)])
def test_argmax_tie_takes_smallest_column(shape):
    """Two identical columns in the same lane position of tiles far apart
    (other CTAs) carry the row maximum: bitwise equal logits, and the
    smaller column must win in every row."""
    K, N, g = 512, 4096, 64
    mat = synth.Matrix("w", synth.AFFINE2, K, N, g, "f16", sigma_scale=0.01)
    (codes, scales, biases), xb = synth.gen_matrix(mat, 21, rows=8)
    xb = xb & np.uint16(0x7FFF)                              # positive activations
    a, b = 16 * 3 + 5, 16 * 250 + 5
    for col in (b, a):                                       # w = 0.05 * 3 + 0.05
        codes[col] = 0xFFFFFFFF
        scales[col] = np.float16(0.05).view(np.uint16)
        biases[col] = np.float16(0.05).view(np.uint16)
    c = Case(synth.AFFINE2, K, N, g, "f16", seed=21, parts=(codes, scales, biases), xb=xb)
    if shape:
        c.plan.set_shape(*shape)
    for M in (1, 8):
        Y, idx, val = c.fused(M, AMAX)
        assert np.array_equal(Y[:M, a], Y[:M, b])
        assert np.all(Y[:M, a] > np.delete(Y[:M], [a, b], axis=1).max(axis=1))
        assert np.all(idx[:M] == a), idx
        _, idx2, _ = c.fused(M, AMAX, want_y=False)
        assert np.all(idx2[:M] == a)


# ----------------------------------------------------------------------------
# arguments

def test_fused_argument_errors():
    c = Case(synth.AFFINE2, 512, 64, 128, "f16", seed=1)
    Y = torch.zeros((8, 64), dtype=torch.float32, device="cuda")
    idx = torch.zeros(8, dtype=torch.int32, device="cuda")

    def status(**kw):
        args = dict(Y=Y, idx=idx, workspace=c.ws)
        args.update(kw)
        ops = args.pop("ops")
        try:
            lbv.verify_fused(c.plan, c.X, 8, c.Wp, ops, **args)
        except lbv.LbvError as e:
            return e.status
        return lbv.OK

    assert status(ops=0x4) == lbv.ERR_INVALID_ARG
    assert status(ops=ROT, Y=None) == lbv.ERR_INVALID_ARG
    assert status(ops=AMAX, idx=None) == lbv.ERR_INVALID_ARG
    assert status(ops=AMAX, workspace=None) == lbv.ERR_WORKSPACE
    assert status(ops=AMAX, workspace=c.ws[:64]) == lbv.ERR_WORKSPACE
    big = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert status(ops=AMAX, workspace=big[8:]) == lbv.ERR_WORKSPACE     # misaligned
    assert status(ops=ROT) == lbv.OK
    assert status(ops=0) == lbv.OK                                       # plain verify
    torch.cuda.synchronize()
    q = Case(synth.Q4_0, 96, 32, 32, "f16", seed=2)                     # K % 128 != 0
    with pytest.raises(lbv.LbvError) as e:
        lbv.verify_fused(q.plan, q.X, 1, q.Wp, ROT, Y=torch.zeros((8, 32), device="cuda"))
    assert e.value.status == lbv.ERR_UNSUPPORTED
    t = Case(synth.AFFINE2, 512, 256, 128, "f16", seed=1, flags=lbv.PLAN_TCGEN05)
    with pytest.raises(lbv.LbvError) as e:
        lbv.verify_fused(t.plan, t.X, 1, t.Wp, AMAX, idx=idx, workspace=t.ws)
    assert e.value.status == lbv.ERR_UNSUPPORTED


# ----------------------------------------------------------------------------
# the full head, in the benchmark's launch configuration

def test_full_head_fused():
    (mat, parts, xb), = synth.gen_workload("head_rot_affine2_g128_5120x151936")
    K, N = mat.K, mat.N
    plan = lbv.Plan(lbv.FMT_AFFINE2, K, N, mat.group, DT[mat.xdtype], lbv.PLAN_PDL)
    Wp = dev(lbv.pack(lbv.FMT_AFFINE2, parts, K, N, mat.group, plan=plan))
    X = dev(xb.view(np.int16))
    Xr = torch.zeros_like(X)
    lbv.fused_rotation(X, Xr, 8, K, DT[mat.xdtype])
    ws = workspace()
    Y = torch.empty((8, N), dtype=torch.float32, device="cuda")
    Yv = torch.empty((8, N), dtype=torch.float32, device="cuda")
    idx = torch.full((8,), SENT_I, dtype=torch.int32, device="cuda")
    val = torch.zeros(8, dtype=torch.float32, device="cuda")
    idx2 = torch.full((8,), SENT_I, dtype=torch.int32, device="cuda")
    lbv.verify_fused(plan, X, 8, Wp, ROT | AMAX, Y=Y, idx=idx, val=val, workspace=ws)
    lbv.verify_fused(plan, X, 8, Wp, ROT | AMAX, idx=idx2, workspace=ws)
    lbv.verify_gemm(plan, Xr, 8, Wp, Yv)
    torch.cuda.synchronize()
    plan.device_status()
    Yg, Yvg = Y.cpu().numpy(), Yv.cpu().numpy()
    ig, vg = idx.cpu().numpy(), val.cpu().numpy()
    assert np.array_equal(Yg, Yvg)
    assert np.array_equal(ig, first_argmax(Yg))
    assert np.array_equal(idx2.cpu().numpy(), ig)
    assert np.array_equal(vg.view(np.uint32), Yg[np.arange(8), ig].view(np.uint32))
    # the oracle on each row's 16 largest GPU logits and sampled columns
    top = np.argsort(-Yg, axis=1)[:, :16]
    rng = np.random.default_rng(0)
    cols = np.unique(np.concatenate([top.ravel(), rng.choice(N, 128, replace=False)]))
    Xf = oracle.x_to_f64(oracle.round_x(oracle.fwht128(oracle.x_to_f64(xb, mat.xdtype)),
                                        mat.xdtype), mat.xdtype)
    Yref, A = oracle.verify(lbv.FMT_AFFINE2, parts, Xf, K, N, mat.group, cols=cols)
    tol = RTOL * A + ATOL
    assert np.all(np.abs(Yg[:, cols] - Yref) <= tol)
    pos = {c: i for i, c in enumerate(cols)}
    for m in range(8):
        j = pos[ig[m]]
        jt = [pos[c] for c in top[m]]
        best = jt[int(np.argmax(Yref[m, jt]))]
        assert Yref[m, j] >= Yref[m, best] - tol[m, j] - tol[m, best]
    assert np.all(ws.cpu().numpy() == 0)
