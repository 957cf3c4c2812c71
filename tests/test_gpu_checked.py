"""The checked build on the GPU.  liblbv_checked.so (LBV_CHECKED) tests, in its
kernels, every copy and buffer range it cannot prove in range by construction
and records a bounds error instead of making the access.  Run in a child
process that loads it (LBV_LIBRARY=checked), small cases of every kernel of the
default path must agree with the oracle and leave the plan's status clean:
every format and dtype, ragged N and K, K splits 2..8, both warp shapes, the
fused head with rotation and argmax, the grouped launch, both 1-row kernels,
and the two tcgen05 kernels over several K splits.  This stands in for a
memory checker, which cannot run here."""
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RTOL, ATOL = 1e-4, 1e-6
SENTINEL = np.float32(-12345.5)

# fmt, K, N, group, xdtype, shape (warps, tiles per warp, splits) or None, flags
CASES = [
    ("sign1_g128", 512, 256, 128, "f16", None, 0),
    ("sign1_g128", 1408, 200, 128, "f16", (16, 1, 2), 0),
    ("sign1_g128", 640, 96, 128, "bf16", (8, 4, 1), 0),
    ("affine2", 768, 136, 64, "bf16", (16, 2, 3), 0),
    ("affine2", 640, 40, 128, "f16", (16, 1, 5), 0),
    ("affine2", 352, 56, 32, "f16", (8, 2, 8), 0),
    ("affine2", 384, 33, 128, "bf16", None, 0),
    ("q4_0", 800, 72, 32, "f16", (8, 4, 2), 0),
    ("q4_0", 1024, 48, 32, "bf16", (16, 2, 4), 0),
    ("sign1_g128", 1024, 80, 128, "f16", None, "gemv"),
    ("affine2", 512, 40, 64, "f16", None, "gemv"),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from few_row_packed_gb300 import buildlib
    import oracle
    buildlib.build(checked=True)
    oracle.build()


def child():
    """Runs in a process with LBV_LIBRARY=checked."""
    import few_row_packed_gb300 as lbv
    import oracle
    import synth
    assert lbv.lib().lbv_checked_build() == 1
    FMT = {"sign1_g128": lbv.FMT_SIGN1_G128, "affine2": lbv.FMT_AFFINE2, "q4_0": lbv.FMT_Q4_0}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n = 0

    def check(Y, M, Yref, A):
        err = np.abs(Y[:M].astype(np.float64) - Yref[:M])
        assert np.all(err <= RTOL * A[:M] + ATOL), (err / (RTOL * A[:M] + ATOL)).max()
        assert np.all(Y[M:] == SENTINEL)

    for fmtname, K, N, group, xd, shape, flags in CASES:
        fmt = FMT[fmtname]
        mat = synth.Matrix("w", fmtname, K, N, group, xd)
        parts, xb = synth.gen_matrix(mat, 3)
        pf = lbv.PLAN_PDL | (lbv.PLAN_FORCE_GEMV if flags == "gemv" else 0)
        P = lbv.Plan(fmt, K, N, group, lbv.DTYPE_BY_NAME[xd], pf)
        if shape:
            P.set_shape(*shape)
        Wp = dev(lbv.pack(fmt, parts, K, N, group, plan=P))
        X = dev(xb.view(np.int16))
        Yref, A = oracle.verify(fmt, parts, oracle.x_to_f64(xb, xd), K, N, group)
        for M in (1, 5, 8):
            Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
            lbv.verify_gemm(P, X, M, Wp, Y)
            torch.cuda.synchronize()
            P.device_status()
            check(Y.cpu().numpy(), M, Yref, A)
            n += 1

    # the tcgen05 kernels (fp16 operands: every format; e4m3: the g128 formats),
    # every K split whose shape fits
    TC = [("sign1_g128", 2048, 520, 128, "f16", lbv.PLAN_TCGEN05, (1, 2, 3, 6)),
          ("affine2", 1536, 260, 32, "f16", lbv.PLAN_TCGEN05, (1, 4)),
          ("q4_0", 1024, 400, 32, "f16", lbv.PLAN_TCGEN05, (2, 8)),
          ("sign1_g128", 2048, 520, 128, "f16", lbv.PLAN_TC_E4M3, (1, 2, 4, 8)),
          ("affine2", 2048, 300, 128, "bf16", lbv.PLAN_TC_E4M3, (1, 2, 4))]
    for fmtname, K, N, group, xd, flag, splits in TC:
        fmt = FMT[fmtname]
        mat = synth.Matrix("t", fmtname, K, N, group, xd)
        parts, xb = synth.gen_matrix(mat, 6)
        P = lbv.Plan(fmt, K, N, group, lbv.DTYPE_BY_NAME[xd], lbv.PLAN_PDL | flag)
        Wp = dev(lbv.pack(fmt, parts, K, N, group, plan=P))
        X = dev(xb.view(np.int16))
        Yref, A = oracle.verify(fmt, parts, oracle.x_to_f64(xb, xd), K, N, group)
        ran = 0
        for s in splits:
            try:
                P.set_shape(0, 0, s, 0)
            except lbv.LbvError:
                continue
            for M in (1, 8):
                Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
                lbv.verify_gemm(P, X, M, Wp, Y)
                torch.cuda.synchronize()
                P.device_status()
                check(Y.cpu().numpy(), M, Yref, A)
                n += 1
            ran += 1
        assert ran > 0, (fmtname, flag)

    # fused head: rotation in the prologue, logits and argmax
    K, N = 1024, 200
    mat = synth.Matrix("h", "affine2", K, N, 128, "f16", rotate=True)
    parts, xb = synth.gen_matrix(mat, 4)
    P = lbv.Plan(lbv.FMT_AFFINE2, K, N, 128, lbv.F16, lbv.PLAN_PDL)
    Wp = dev(lbv.pack(lbv.FMT_AFFINE2, parts, K, N, 128, plan=P))
    X = dev(xb.view(np.int16))
    Xr = torch.empty_like(X)
    lbv.fused_rotation(X, Xr, 8, K)
    torch.cuda.synchronize()
    xr = Xr.cpu().numpy().view(np.uint16)
    Yref, A = oracle.verify(lbv.FMT_AFFINE2, parts, oracle.x_to_f64(xr, "f16"), K, N, 128)
    ws = torch.zeros(lbv.fused_workspace_bytes(), dtype=torch.uint8, device="cuda")
    idx = torch.full((8,), -7, dtype=torch.int32, device="cuda")
    for M in (1, 8):
        Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
        lbv.verify_fused(P, X, M, Wp, lbv.FUSED_ROTATE | lbv.FUSED_ARGMAX, Y=Y, idx=idx,
                         workspace=ws)
        torch.cuda.synchronize()
        P.device_status()
        got = Y.cpu().numpy()
        check(got, M, Yref, A)
        assert np.array_equal(idx.cpu().numpy()[:M], got[:M].argmax(axis=1))
        n += 1

    # grouped launch over independent problems, one of them inactive
    shapes = [(512, 64), (384, 48), (640, 32)]
    G = lbv.Group(lbv.FMT_Q4_0, 32, lbv.F16, shapes, lbv.PLAN_PDL)
    probs, refs = [], []
    for i, ((K, N), M) in enumerate(zip(shapes, (3, 8, 0))):
        mat = synth.Matrix("g", "q4_0", K, N, 32, "f16")
        parts, xb = synth.gen_matrix(mat, 10 + i)
        Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
        probs.append((dev(xb.view(np.int16)), M, dev(lbv.pack(lbv.FMT_Q4_0, parts, K, N, 32)), Y))
        refs.append(oracle.verify(lbv.FMT_Q4_0, parts, oracle.x_to_f64(xb, "f16"), K, N, 32))
    lbv.verify_grouped(G, probs)
    torch.cuda.synchronize()
    G.device_status()
    for (X, M, W, Y), (Yref, A) in zip(probs, refs):
        got = Y.cpu().numpy()
        if M:
            check(got, M, Yref, A)
        else:
            assert np.all(got == SENTINEL)
        n += 1
    print(f"checked build: {n} calls agree with the oracle, status clean")


def test_checked_build_parity():
    env = dict(os.environ, LBV_LIBRARY="checked", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", "import tests.test_gpu_checked as t; t.child()"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "status clean" in r.stdout
