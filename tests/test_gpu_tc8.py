"""GPU tests of plans created with PLAN_TC_E4M3: the e4m3 tensor-memory kernel
and the record layout it reads, against the fp64 oracle (the same tolerance as
every verify path: 1e-4 * sum_k |x_k w_k| + 1e-6 per element; dequantized
weights bit for bit, through the kernel's own e4m3 decode)."""
import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import oracle
import synth
import test_gpu_fused as F
from test_gpu_parity import ATOL, DT, FMT, RTOL, SENTINEL, Case, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
T8 = lbv.PLAN_TC_E4M3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


# ----------------------------------------------------------------------------
# The layout, read back from its written specification (t8_layout.h): one
# record per (128-column tile, 128-K group, quarter), in the order
# ((tile * ngroups + group) * 4 + quarter): codes [CB/16][32 columns][16
# bytes], then side [32 columns][SB bytes].  Word i of a column holds, for
# 2-bit codes, k = 16i + 4j + b at bit 8b + 2j; for 1-bit codes,
# k = 32i + 4j + b at bit 8b + j.

SPEC = {lbv.FMT_SIGN1_G128: (16, 2, 1), lbv.FMT_AFFINE2: (32, 4, 2)}   # CB, SB, W


def read_layout(fmt, packed, K, N):
    cb, sb, W = SPEC[fmt]
    nt, ng = -(-N // 128), K // 128
    recs = packed.reshape(nt, ng, 4, 32 * (cb + sb)).transpose(0, 2, 1, 3)   # [tile][q][g]
    codes = np.ascontiguousarray(recs[..., :32 * cb]).reshape(nt, 4, ng, cb // 16, 32, 16)
    words = np.ascontiguousarray(codes.transpose(0, 1, 2, 4, 3, 5)).reshape(
        nt, 4, ng, 32, cb).view(np.uint32)                  # [tile][q][g][lane][word]
    out = np.zeros((nt * 128, K), np.int64)
    for k in range(128):
        if W == 2:
            i, j, b = k // 16, (k % 16) // 4, k % 4
            bit = 8 * b + 2 * j
        else:
            i, j, b = k // 32, (k % 32) // 4, k % 4
            bit = 8 * b + j
        v = (words[..., i] >> np.uint32(bit)) & ((1 << W) - 1)       # [tile][q][g][lane]
        out[:, k::128] = v.transpose(0, 1, 3, 2).reshape(nt * 128, ng)
    side = np.ascontiguousarray(recs[..., 32 * cb:]).view(np.uint16).reshape(nt, 4, ng, 32, -1)
    side = side.transpose(0, 1, 3, 2, 4).reshape(nt * 128, ng, -1)
    return out, side


def canonical_codes(fmt, parts, K, N):
    w = parts[0]
    if fmt == lbv.FMT_SIGN1_G128:
        return ((w[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(N, K)
    return ((w[:, :, None] >> (2 * np.arange(16, dtype=np.uint32))) & 3).reshape(N, K)


@pytest.mark.parametrize("fmtname,K,N", [(synth.SIGN1_G128, 512, 48), (synth.SIGN1_G128, 384, 150),
                                         (synth.AFFINE2, 384, 140), (synth.AFFINE2, 256, 33)])
def test_t8_pack_is_lossless(fmtname, K, N):
    fmt = FMT[fmtname]
    mat = synth.Matrix("w", fmtname, K, N, 128, "f16")
    parts, _ = synth.gen_matrix(mat, 13, rows=1)
    plan = lbv.Plan(fmt, K, N, 128, lbv.F16, T8)
    packed = plan.pack(parts)
    cb, sb, _ = SPEC[fmt]
    assert packed.size == plan.packed_bytes == -(-N // 128) * 4 * (K // 128) * 32 * (cb + sb)
    codes, side = read_layout(fmt, packed, K, N)
    assert np.array_equal(codes[:N], canonical_codes(fmt, parts, K, N))
    assert np.all(codes[N:] == 0) and np.all(side[N:] == 0)
    assert np.array_equal(side[:N, :, 0], parts[1])
    if fmt == lbv.FMT_AFFINE2:
        assert np.array_equal(side[:N, :, 1], parts[2])


def test_t8_plan_kernel_shape_and_errors():
    plan = lbv.Plan(lbv.FMT_SIGN1_G128, 1024, 256, 128, lbv.F16, T8)
    for M in (1, 8):
        assert plan.query(M)[0] == lbv.KERNEL_FEWROW_TC8
    w, t, s, c = plan.shape()
    assert (w, t) == (0, 0) and s in (1, 2, 4, 8) and c >= 1
    for s in (1, 2, 4, 8):
        plan.set_shape(0, 0, s, 0)
        assert plan.shape()[2] == s
    for bad in (3, 5, 9):
        with pytest.raises(lbv.LbvError):
            plan.set_shape(0, 0, bad, 0)
    for flags in (lbv.PLAN_FORCE_GEMV, lbv.PLAN_TCGEN05, lbv.PLAN_TEST_WAIT_LIMIT):
        with pytest.raises(lbv.LbvError) as e:
            lbv.Plan(lbv.FMT_SIGN1_G128, 512, 256, 128, lbv.F16, T8 | flags)
        assert e.value.status == lbv.ERR_INVALID_ARG
    for fmt, group in ((lbv.FMT_AFFINE2, 64), (lbv.FMT_AFFINE2, 32), (lbv.FMT_Q4_0, 32)):
        with pytest.raises(lbv.LbvError) as e:
            lbv.Plan(fmt, 512, 256, group, lbv.F16, T8)
        assert e.value.status == lbv.ERR_UNSUPPORTED


@pytest.mark.parametrize("fmtname,K,N", [(synth.SIGN1_G128, 640, 200), (synth.AFFINE2, 512, 130),
                                         (synth.AFFINE2, 1024, 300)])
def test_t8_dequant_bit_exact(fmtname, K, N):
    """The kernel's decode (LOP3 fields read as e4m3 bytes, times 2^(9 - f))
    gives back every code: the dense dequant equals the oracle's bit for bit."""
    mat = synth.Matrix("w", fmtname, K, N, 128, "f16", sigma_scale=0.01)
    parts, _ = synth.gen_matrix(mat, 6, rows=1)
    fmt = FMT[fmtname]
    plan = lbv.Plan(fmt, K, N, 128, lbv.F16, T8)
    Wp = dev(plan.pack(parts))
    W = torch.zeros((K, N), dtype=torch.int16, device="cuda")
    lbv.dequant_fp16(plan, Wp, W)
    torch.cuda.synchronize()
    assert np.array_equal(W.cpu().numpy().view(np.uint16), oracle.dequant_f16(fmt, parts, K, N, 128))


SMALL = [
    # fmt, K, N, xdtype
    (synth.SIGN1_G128, 512, 256, "f16"),
    (synth.SIGN1_G128, 1408, 200, "f16"),    # ragged N tail
    (synth.SIGN1_G128, 640, 96, "bf16"),
    (synth.SIGN1_G128, 128, 33, "f16"),      # one group
    (synth.AFFINE2, 640, 40, "f16"),
    (synth.AFFINE2, 384, 33, "bf16"),
    (synth.AFFINE2, 1024, 600, "f16"),       # several tiles per warpgroup
    (synth.AFFINE2, 2048, 130, "bf16"),
]


@pytest.mark.parametrize("fmtname,K,N,xdtype", SMALL)
def test_t8_parity_small_all_M(fmtname, K, N, xdtype):
    c = Case(fmtname, K, N, 128, xdtype, seed=0, flags=T8)
    for M in range(1, 9):
        c.check(c.run(M), M)


@pytest.mark.parametrize("fmtname,K,N,xdtype", [
    (synth.SIGN1_G128, 2048, 520, "f16"), (synth.AFFINE2, 2048, 300, "bf16"),
    (synth.AFFINE2, 1024, 1100, "f16")])
def test_t8_split_k_and_cluster_shapes(fmtname, K, N, xdtype):
    """Every K split (cluster size 1, 2, 4, 8) with several cluster counts,
    including clusters that own fewer tiles than warpgroups: within
    tolerance, and each shape deterministic."""
    c = Case(fmtname, K, N, 128, xdtype, seed=3, flags=T8)
    tried = 0
    for splits in (1, 2, 4, 8):
        for ctas in (0, 1, 3, 7):
            try:
                c.plan.set_shape(0, 0, splits, ctas)
            except lbv.LbvError:
                continue
            tried += 1
            for M in (1, 5, 8):
                Y = c.run(M)
                c.check(Y, M)
                assert np.array_equal(Y, c.run(M))
    assert tried >= 10


def test_t8_rows_independent_bitwise():
    c = Case(synth.AFFINE2, 1024, 260, 128, "f16", seed=4, flags=T8)
    Y8 = c.run(8)
    for M in (1, 3, 7):
        assert np.array_equal(c.run(M)[:M], Y8[:M])
    X2 = c.X.clone()
    X2[5:] = 0
    assert np.array_equal(c.run(5, X=X2)[:5], Y8[:5])


def wide_range_rows(K, xdtype, seed):
    """Activation rows that stress the per-row power-of-two scale and the
    three-term e4m3 split: tiny, huge, zero, mixed magnitudes, subnormals."""
    rng = np.random.default_rng(seed)
    big = 6.0e4 if xdtype == "f16" else 1.0e30
    tiny = 2.0 ** -23 if xdtype == "f16" else 2.0 ** -120
    rows = [
        rng.standard_normal(K) * 1e-3,
        np.clip(rng.standard_normal(K) * big / 8, -big, big),
        np.zeros(K),
        np.sign(rng.standard_normal(K)) * 2.0 ** rng.uniform(-20, 14, K),
        rng.standard_normal(K) * tiny,
        np.where(rng.random(K) < 0.01, big, rng.standard_normal(K) * 1e-2),
        rng.standard_normal(K),
        np.full(K, -1.0),
    ]
    X = np.stack(rows)
    if xdtype == "f16":
        return X.astype(np.float16).view(np.uint16)
    return (X.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("fmtname,xdtype", [(synth.SIGN1_G128, "f16"), (synth.AFFINE2, "f16"),
                                            (synth.AFFINE2, "bf16"), (synth.SIGN1_G128, "bf16")])
def test_t8_wide_range_activations(fmtname, xdtype):
    K, N = 1024, 260
    c = Case(fmtname, K, N, 128, xdtype, seed=8, flags=T8)
    xb = wide_range_rows(K, xdtype, 8)
    X = dev(xb.view(np.int16))
    Yref, A = oracle.verify(c.fmt, c.parts, oracle.x_to_f64(xb, xdtype), K, N, 128)
    for M in (1, 8):
        Y = c.run(M, X=X)
        err = np.abs(Y[:M].astype(np.float64) - Yref[:M])
        tol = RTOL * A[:M] + ATOL
        assert np.all(err <= tol), f"M={M}: worst {(err / tol).max():.3g}x tol"
        assert np.all(Y[M:] == SENTINEL)


@pytest.mark.parametrize("dx", [0, 1, 8])
def test_t8_strided_x(dx):
    """X with a row stride ldx = K + dx and X one element into its buffer
    (dx odd): the plain-load staging path."""
    K, N = 768, 300
    c = Case(synth.AFFINE2, K, N, 128, "f16", seed=5, flags=T8)
    base = torch.zeros((8 * (K + dx) + 8,), dtype=torch.int16, device="cuda")
    off = 1 if dx % 2 else 0
    Xs = base[off:off + 8 * (K + dx)].view(8, K + dx)
    Xs[:, :K] = c.X
    for M in (1, 8):
        Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
        lbv.verify_gemm(c.plan, Xs, M, c.Wp, Y, ldx=K + dx)
        torch.cuda.synchronize()
        c.plan.device_status()
        c.check(Y.cpu().numpy(), M)


# ----------------------------------------------------------------------------
# fused head on the e4m3 kernel

@pytest.mark.parametrize("fmtname,K,N,xdtype,signs", [
    (synth.AFFINE2, 1280, 400, "f16", False),
    (synth.AFFINE2, 1280, 400, "f16", True),
    (synth.AFFINE2, 768, 2000, "bf16", True),
    (synth.SIGN1_G128, 1024, 200, "f16", False)])
def test_t8_fused_rotate_and_argmax(fmtname, K, N, xdtype, signs):
    c = F.Case(fmtname, K, N, 128, xdtype, seed=K + N, flags=T8, signs=signs)
    Yref, A = c.oracle_y(rotate=True)
    Xr = c.exported_x()
    for M in range(1, 9):
        Y, idx, val = c.fused(M, F.ROT)
        assert np.all(idx == F.SENT_I), "argmax written without the op"
        assert np.array_equal(Y, c.verify(M, Xr)), "fused rotation differs from the exported one"
        err = np.abs(Y[:M].astype(np.float64) - Yref[:M])
        assert np.all(err <= RTOL * A[:M] + ATOL), f"M={M}: worst {(err / (RTOL * A[:M] + ATOL)).max():.3g}x tol"
        assert np.all(Y[M:] == F.SENT_Y)
        Y2, idx2, val2 = c.fused(M, F.ROT | F.AMAX)
        assert np.array_equal(Y2, Y)
        F.check_argmax(Y2, idx2, val2, M, Yref, A, N)
        _, idx3, _ = c.fused(M, F.ROT | F.AMAX, want_y=False)
        assert np.array_equal(idx3, idx2)
    assert np.all(c.ws.cpu().numpy() == 0), "workspace not left zeroed"


def test_t8_fused_split_shapes():
    c = F.Case(synth.AFFINE2, 2048, 1000, 128, "f16", seed=9, flags=T8, signs=True)
    Yref, A = c.oracle_y(rotate=True)
    Xr = c.exported_x()
    tried = 0
    for splits in (1, 2, 4, 8):
        for ctas in (0, 3):
            try:
                c.plan.set_shape(0, 0, splits, ctas)
            except lbv.LbvError:
                continue
            tried += 1
            for M in (1, 8):
                Y, idx, val = c.fused(M, F.ROT | F.AMAX)
                assert np.array_equal(Y, c.verify(M, Xr))
                assert np.all(np.abs(Y[:M] - Yref[:M]) <= RTOL * A[:M] + ATOL)
                F.check_argmax(Y, idx, val, M, Yref, A, c.N)
    assert tried >= 6


def test_t8_argmax_tie_takes_smallest_column():
    """Two identical columns in different tiles (owned by different CTAs)
    carry the row maximum: the smaller column wins."""
    K, N = 512, 4096
    mat = synth.Matrix("w", synth.AFFINE2, K, N, 128, "f16", sigma_scale=0.01)
    (codes, scales, biases), xb = synth.gen_matrix(mat, 21, rows=8)
    xb = xb & np.uint16(0x7FFF)
    a, b = 128 * 3 + 5, 128 * 25 + 5
    for col in (b, a):
        codes[col] = 0xFFFFFFFF
        scales[col] = np.float16(0.05).view(np.uint16)
        biases[col] = np.float16(0.05).view(np.uint16)
    c = F.Case(synth.AFFINE2, K, N, 128, "f16", seed=21, flags=T8, parts=(codes, scales, biases),
               xb=xb)
    for splits in (1, 2, 4):
        c.plan.set_shape(0, 0, splits, 0)
        for M in (1, 8):
            Y, idx, val = c.fused(M, F.AMAX)
            assert np.array_equal(Y[:M, a], Y[:M, b])
            assert np.all(idx[:M] == a), idx
