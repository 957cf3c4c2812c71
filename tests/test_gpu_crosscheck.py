"""Second references and guards for the CUDA path (through the C ABI):

- an independent library: cuBLAS fp32 matmul (torch, TF32 off) of X and the
  exact weights the oracle unpacks, on the GPU.  Both it and the kernel sit
  within the verify tolerance of the exact result, so they agree within twice
  that tolerance;
- row permutation: permuting X's rows permutes Y's rows, bit for bit;
- guard bytes around Y, the argmax outputs and the fused head's workspace
  stay untouched.
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
SENT = -12345.5
GUARD = 0xA5

CASES = [
    # fmt, K, N, group, xdtype
    (synth.SIGN1_G128, 1408, 200, 128, "f16"),
    (synth.SIGN1_G128, 2048, 96, 128, "bf16"),
    (synth.AFFINE2, 768, 136, 64, "bf16"),
    (synth.AFFINE2, 1280, 80, 128, "f16"),
    (synth.AFFINE2, 352, 56, 32, "f16"),
    (synth.Q4_0, 1088, 72, 32, "f16"),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def setup(fmtname, K, N, group, xdtype, seed):
    mat = synth.Matrix("w", fmtname, K, N, group, xdtype,
                       sigma_scale=0.02 if fmtname == synth.SIGN1_G128 else 0.01)
    parts, xb = synth.gen_matrix(mat, seed, rows=8)
    plan = lbv.Plan(FMT[fmtname], K, N, group, DT[xdtype])
    Wp = dev(lbv.pack(FMT[fmtname], parts, K, N, group, plan=plan))
    return parts, xb, plan, Wp


def run(plan, X, M, Wp, N):
    Y = torch.full((8, N), SENT, dtype=torch.float32, device="cuda")
    lbv.verify_gemm(plan, X, M, Wp, Y)
    torch.cuda.synchronize()
    plan.device_status()
    return Y.cpu().numpy()


@pytest.mark.parametrize("fmtname,K,N,group,xdtype", CASES)
def test_cublas_fp32_crosscheck(fmtname, K, N, group, xdtype):
    parts, xb, plan, Wp = setup(fmtname, K, N, group, xdtype, seed=11)
    Y = run(plan, dev(xb.view(np.int16)), 8, Wp, N)
    Xf = oracle.x_to_f64(xb, xdtype)
    W = oracle.unpack(FMT[fmtname], parts, K, N, group)       # exact weights (fp64)
    prev = torch.get_float32_matmul_precision()
    torch.set_float32_matmul_precision("highest")             # plain fp32, no TF32
    try:
        Yt = (dev(Xf.astype(np.float32)) @ dev(W.astype(np.float32))).cpu().numpy()
    finally:
        torch.set_float32_matmul_precision(prev)
    _, A = oracle.verify(FMT[fmtname], parts, Xf, K, N, group)
    err = np.abs(Y.astype(np.float64) - Yt.astype(np.float64))
    tol = 2 * (RTOL * A + ATOL)
    assert np.all(err <= tol), f"worst {(err / tol).max():.3g}x tol"


@pytest.mark.parametrize("fmtname,K,N,group,xdtype", CASES[::2])
def test_row_permutation_bitwise(fmtname, K, N, group, xdtype):
    parts, xb, plan, Wp = setup(fmtname, K, N, group, xdtype, seed=12)
    perm = np.random.default_rng(13).permutation(8)
    Y = run(plan, dev(xb.view(np.int16)), 8, Wp, N)
    Yp = run(plan, dev(xb[perm].view(np.int16)), 8, Wp, N)
    assert np.array_equal(Yp, Y[perm])
    for M in (3, 6):                          # the first M rows of the permuted input
        assert np.array_equal(run(plan, dev(xb[perm].view(np.int16)), M, Wp, N)[:M],
                              Y[perm][:M])


@pytest.mark.parametrize("M", [1, 8])
def test_guard_rows_around_y(M):
    fmtname, K, N, group, xdtype = CASES[3]
    parts, xb, plan, Wp = setup(fmtname, K, N, group, xdtype, seed=14)
    full = torch.full((10, N), SENT, dtype=torch.float32, device="cuda")
    lbv.verify_gemm(plan, dev(xb.view(np.int16)), M, Wp, full[1:9])
    torch.cuda.synchronize()
    got = full.cpu().numpy()
    assert np.all(got[0] == SENT) and np.all(got[1 + M:] == SENT)
    assert np.array_equal(got[1:1 + M], run(plan, dev(xb.view(np.int16)), M, Wp, N)[:M])


def test_guards_around_fused_outputs_and_workspace():
    """Fused head (rotation and argmax): nothing outside Y[:M], idx[:M],
    val[:M] and the workspace is written, and the workspace is left zeroed."""
    K, N, group = 1024, 320, 128
    parts, xb, plan, Wp = setup(synth.AFFINE2, K, N, group, "f16", seed=15)
    X = dev(xb.view(np.int16))
    wsb = lbv.fused_workspace_bytes()
    ws_full = torch.full((wsb + 128,), GUARD, dtype=torch.uint8, device="cuda")
    ws_full[64:64 + wsb] = 0
    for M in (1, 5, 8):
        Y_full = torch.full((10, N), SENT, dtype=torch.float32, device="cuda")
        idx_full = torch.full((10,), -7, dtype=torch.int32, device="cuda")
        val_full = torch.full((10,), SENT, dtype=torch.float32, device="cuda")
        lbv.verify_fused(plan, X, M, Wp, lbv.FUSED_ROTATE | lbv.FUSED_ARGMAX, Y=Y_full[1:9],
                         idx=idx_full[1:9], val=val_full[1:9], workspace=ws_full[64:64 + wsb])
        torch.cuda.synchronize()
        plan.device_status()
        Yg, ig, vg = Y_full.cpu().numpy(), idx_full.cpu().numpy(), val_full.cpu().numpy()
        assert np.all(Yg[0] == SENT) and np.all(Yg[1 + M:] == SENT)
        assert ig[0] == -7 and np.all(ig[1 + M:] == -7)
        assert vg[0] == SENT and np.all(vg[1 + M:] == SENT)
        # the outputs inside are those of the same call: argmax of its own logits
        assert np.array_equal(ig[1:1 + M], np.argmax(Yg[1:1 + M], axis=1))
        assert np.array_equal(vg[1:1 + M], Yg[1:1 + M][np.arange(M), ig[1:1 + M]])
        w = ws_full.cpu().numpy()
        assert np.all(w[:64] == GUARD) and np.all(w[64 + wsb:] == GUARD)
        assert np.all(w[64:64 + wsb] == 0), "workspace not left zeroed"
