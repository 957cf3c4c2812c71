"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (plan with programmatic dependent launch), on sampled output
columns that the fp64 oracle computes one by one."""
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


def sample_cols(N, n=192, seed=0):
    rng = np.random.default_rng(seed)
    c = np.concatenate([np.arange(16), np.arange(N - 16, N), rng.choice(N, n, replace=False)])
    return np.unique(c)


def check_matrix(mat, parts, xb, Ms=range(1, 9), rotate=False):
    fmt = FMT[mat.fmt]
    K, N = mat.K, mat.N
    plan = lbv.Plan(fmt, K, N, mat.group, DT[mat.xdtype], lbv.PLAN_PDL)
    Wp = torch.from_numpy(lbv.pack(fmt, parts, K, N, mat.group)).cuda()
    X = torch.from_numpy(xb.view(np.int16)).cuda()
    Xf = oracle.x_to_f64(xb, mat.xdtype)
    if rotate:
        Xr = torch.zeros_like(X)
        lbv.fwht128(X, Xr, 8, K, DT[mat.xdtype])
        X = Xr
        Xf = oracle.x_to_f64(oracle.round_x(oracle.fwht128(Xf), mat.xdtype), mat.xdtype)
    cols = sample_cols(N)
    Yref, A = oracle.verify(fmt, parts, Xf, K, N, mat.group, cols=cols)
    for M in Ms:
        Y = torch.full((8, N), -7.0, dtype=torch.float32, device="cuda")
        lbv.verify_gemm(plan, X, M, Wp, Y)
        torch.cuda.synchronize()
        plan.device_status()          # no bounded wait gave up
        got = Y.cpu().numpy()
        err = np.abs(got[:M][:, cols] - Yref[:M])
        tol = RTOL * A[:M] + ATOL
        assert np.all(err <= tol), f"{mat.name} M={M}: worst {(err / tol).max():.3g}x tol"
        assert np.all(got[M:] == -7.0)
        assert np.all(np.isfinite(got[:M]))


@pytest.mark.parametrize("name", ["sign1_tiny_512x256", "sign1_mlp_up_5120x17408",
                                  "affine2_g64_6144x6144", "affine2_g64_kv_5120x1024"])
def test_full_config(name):
    for mat, parts, xb in synth.gen_workload(name):
        check_matrix(mat, parts, xb)


def test_full_rotated_head():
    (mat, parts, xb), = synth.gen_workload("head_rot_affine2_g128_5120x151936")
    check_matrix(mat, parts, xb, rotate=True)


def test_full_q4_0_stack():
    for i, (mat, parts, xb) in enumerate(synth.gen_workload("q4_0_stack_4x7")):
        check_matrix(mat, parts, xb, Ms=(1, 8) if i % 7 else (1, 3, 8))
