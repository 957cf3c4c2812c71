"""GPU tests of plans created with PLAN_TCGEN05: the tcgen05 few-row kernel and
the 128-column record layout it reads, against the fp64 oracle (same tolerance
as the default kernel: 1e-4 * sum_k |x_k w_k| + 1e-6 per element; dequantized
weights bit for bit)."""
import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import oracle
import synth
from test_gpu_parity import ATOL, DT, FMT, RTOL, SENTINEL, SMALL, Case, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
TC = lbv.PLAN_TCGEN05


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lbv.build()
    oracle.build()


# ----------------------------------------------------------------------------
# The tcgen05 layout, read back from its written specification (tc_layout.h):
# one record per (128-column tile, chunk) in tile-major order: codes
# [CB/16][128 columns][16 bytes], then side [128 columns][SB bytes].  The CB
# bytes of column c are words j; word j holds pairs p = PPW*j + s: the code of
# k = 2p at bit s*W and of k = 2p + 1 at bit 16 + s*W.

SPEC = {  # fmt: group -> (chunk_k, code bytes CB, side bytes SB, bits W)
    lbv.FMT_SIGN1_G128: {128: (128, 16, 2, 1)},
    lbv.FMT_AFFINE2: {32: (64, 16, 8, 2), 64: (64, 16, 4, 2), 128: (128, 32, 4, 2)},
    lbv.FMT_Q4_0: {32: (64, 32, 4, 4)},
}


def read_layout(fmt, packed, K, N, group):
    ck, cb, sb, W = SPEC[fmt][group]
    ppw = 16 // W
    ntiles, nch = -(-N // 128), -(-K // ck)
    rec = 128 * (cb + sb)
    recs = packed.reshape(ntiles, nch, rec)
    codes = np.ascontiguousarray(recs[:, :, :128 * cb]).reshape(ntiles, nch, cb // 16, 128, 16)
    words = np.ascontiguousarray(codes.transpose(0, 1, 3, 2, 4)).reshape(
        ntiles, nch, 128, cb).view(np.uint32)                    # [tile][chunk][col][word]
    out = np.full((ntiles * 128, nch * ck), -1, np.int64)
    mask = (1 << W) - 1
    n = (np.arange(ntiles)[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
    for j in range(cb // 4):
        for s_ in range(ppw):
            p = ppw * j + s_
            for h in range(2):
                v = (words[:, :, :, j] >> np.uint32(s_ * W + 16 * h)) & mask   # [tile][chunk][col]
                k = np.arange(nch) * ck + 2 * p + h
                out[np.ix_(n, k)] = v.transpose(0, 2, 1).reshape(ntiles * 128, nch)
    side = np.ascontiguousarray(recs[:, :, 128 * cb:]).view(np.uint16).reshape(ntiles, nch, 128, -1)
    return out, side


def canonical_codes(fmt, parts, K, N):
    if fmt == lbv.FMT_SIGN1_G128:
        w = parts[0]
        return ((w[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(N, K)
    if fmt == lbv.FMT_AFFINE2:
        w = parts[0]
        return ((w[:, :, None] >> (2 * np.arange(16, dtype=np.uint32))) & 3).reshape(N, K)
    qs = parts[0][:, :, 2:]
    return np.concatenate([qs & 15, qs >> 4], axis=2).reshape(N, K)




@pytest.mark.parametrize("fmtname,K,N,group", [
    (synth.SIGN1_G128, 512, 48, 128), (synth.SIGN1_G128, 384, 150, 128),
    (synth.AFFINE2, 256, 32, 64), (synth.AFFINE2, 320, 17, 32), (synth.AFFINE2, 384, 140, 128),
    (synth.Q4_0, 192, 32, 32), (synth.Q4_0, 96, 9, 32)])
def test_tc_pack_is_lossless(fmtname, K, N, group):
    fmt = FMT[fmtname]
    mat = synth.Matrix("w", fmtname, K, N, group, "f16")
    parts, _ = synth.gen_matrix(mat, 13, rows=1)
    plan = lbv.Plan(fmt, K, N, group, lbv.F16, TC)
    packed = plan.pack(parts)
    ck = SPEC[fmt][group][0]
    assert packed.size == plan.packed_bytes == -(-N // 128) * -(-K // ck) * 128 * sum(SPEC[fmt][group][1:3])
    codes, side = read_layout(fmt, packed, K, N, group)
    assert np.array_equal(codes[:N, :K], canonical_codes(fmt, parts, K, N))
    assert np.all(codes[N:, :] == 0) and np.all(codes[:, K:] == 0)
    gk = group if fmt == lbv.FMT_AFFINE2 else (128 if fmt == lbv.FMT_SIGN1_G128 else 32)
    per = 2 if fmt == lbv.FMT_AFFINE2 else 1
    for tile in range(side.shape[0]):
        for ch in range(side.shape[1]):
            for c in range(128):
                n = tile * 128 + c
                for j in range(ck // gk):
                    grp = ch * (ck // gk) + j
                    e = side[tile, ch, c, per * j]
                    if n >= N or grp * gk >= K:
                        assert e == 0
                    elif fmt == lbv.FMT_Q4_0:
                        blk = parts[0][n, grp]
                        assert e == int(blk[0]) | (int(blk[1]) << 8)
                    else:
                        assert e == parts[1][n, grp]
                        if fmt == lbv.FMT_AFFINE2:
                            assert side[tile, ch, c, per * j + 1] == parts[2][n, grp]


def test_tc_plan_reports_its_kernel():
    plan = lbv.Plan(lbv.FMT_SIGN1_G128, 512, 256, 128, lbv.F16, TC)
    for M in (1, 8):
        assert plan.query(M)[0] == lbv.KERNEL_FEWROW_TC
    w, t, s, c = plan.shape()
    assert (w, t) == (0, 0) and 1 <= s <= 8 and c >= 1
    with pytest.raises(lbv.LbvError):
        lbv.Plan(lbv.FMT_SIGN1_G128, 512, 256, 128, lbv.F16, TC | lbv.PLAN_FORCE_GEMV)


@pytest.mark.parametrize("fmtname,K,N,group,xdtype", SMALL)
def test_tc_parity_small_all_M(fmtname, K, N, group, xdtype):
    c = Case(fmtname, K, N, group, xdtype, seed=0, flags=TC)
    for M in range(1, 9):
        c.check(c.run(M), M)


@pytest.mark.parametrize("fmtname,K,N,group,xdtype", [
    (synth.SIGN1_G128, 2048, 520, 128, "f16"), (synth.AFFINE2, 2048, 300, 64, "bf16"),
    (synth.AFFINE2, 1536, 260, 32, "f16"), (synth.Q4_0, 1024, 400, 32, "f16")])
def test_tc_split_k_and_cluster_shapes(fmtname, K, N, group, xdtype):
    """Every K split (cluster size) and a few cluster counts, including ones
    that leave a CTA fewer tiles than warpgroups (warpgroup split of K)."""
    c = Case(fmtname, K, N, group, xdtype, seed=3, flags=TC)
    first = None
    for splits in range(1, 9):
        for ctas in (0, 1, 3):
            try:
                c.plan.set_shape(0, 0, splits, ctas)
            except lbv.LbvError:
                continue
            Y = c.run(8)
            c.check(Y, 8)
            if first is None:
                first = Y
    assert first is not None


def test_tc_rows_independent_bitwise():
    c = Case(synth.AFFINE2, 1024, 260, 64, "f16", seed=4, flags=TC)
    Y8 = c.run(8)
    for M in (1, 3, 7):
        assert np.array_equal(c.run(M)[:M], Y8[:M])
    X2 = c.X.clone()
    X2[5:] = 0
    assert np.array_equal(c.run(5, X=X2)[:5], Y8[:5])


@pytest.mark.parametrize("fmtname,K,N,group", [
    (synth.SIGN1_G128, 640, 200, 128), (synth.AFFINE2, 384, 150, 32),
    (synth.AFFINE2, 512, 130, 128), (synth.Q4_0, 320, 140, 32)])
def test_tc_dequant_bit_exact(fmtname, K, N, group):
    mat = synth.Matrix("w", fmtname, K, N, group, "f16", sigma_scale=0.01)
    parts, _ = synth.gen_matrix(mat, 6, rows=1)
    fmt = FMT[fmtname]
    plan = lbv.Plan(fmt, K, N, group, lbv.F16, TC)
    Wp = dev(plan.pack(parts))
    W = torch.zeros((K, N), dtype=torch.int16, device="cuda")
    lbv.dequant_fp16(plan, Wp, W)
    torch.cuda.synchronize()
    assert np.array_equal(W.cpu().numpy().view(np.uint16), oracle.dequant_f16(fmt, parts, K, N, group))


def test_tc_rotated_head_small():
    K, N = 1024, 300
    c = Case(synth.AFFINE2, K, N, 128, "f16", seed=9, rotate=True, flags=TC)
    Xr = torch.zeros_like(c.X)
    lbv.fwht128(c.X, Xr, 8, K, lbv.F16)
    xr_bits = oracle.round_x(oracle.fwht128(c.Xf), "f16")
    Yref, A = oracle.verify(c.fmt, c.parts, oracle.f16_to_f64(xr_bits), K, N, 128)
    for M in (1, 8):
        Y = torch.full((8, N), float(SENTINEL), dtype=torch.float32, device="cuda")
        lbv.verify_gemm(c.plan, Xr, M, c.Wp, Y)
        torch.cuda.synchronize()
        c.plan.device_status()
        got = Y.cpu().numpy()[:M].astype(np.float64)
        assert np.all(np.abs(got - Yref[:M]) <= RTOL * A[:M] + ATOL)


def test_tc_full_1bit_mlp_up_sampled():
    """The bench's 1-bit 5120x17408 shape, checked on sampled columns."""
    rng = np.random.default_rng(1)
    cols = np.sort(rng.choice(17408, 256, replace=False))
    c = Case(synth.SIGN1_G128, 5120, 17408, 128, "f16", seed=0, cols=cols, flags=TC | lbv.PLAN_PDL)
    for M in (1, 8):
        c.check(c.run(M), M)
