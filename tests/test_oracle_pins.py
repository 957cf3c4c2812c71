"""Pins of the fp64 CPU oracle against what the pages and mathematics fix.

Nothing here compares the oracle with itself: every check is against a
hand-enumerated case from the format definitions (tests/golden), a closed form,
an invariant, a library routine (numpy, scipy, torch, Python fractions) or
brute force on tiny inputs.  All CPU-only.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = {synth.SIGN1_G128: 0, synth.AFFINE2: 1, synth.Q4_0: 2}


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _hex_array(rows, dtype):
    return np.array([[int(v, 16) for v in r] for r in rows], dtype=dtype)


# ----------------------------------------------------------------------------
# fp16 / bf16 conversions

def test_f16_decode_matches_numpy(oracle_lib):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    got = oracle_lib.f16_to_f64(allbits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_f16_round_matches_numpy(oracle_lib):
    rng = np.random.default_rng(1)
    rand = rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000)
    h = np.arange(1, 0x7BFF, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2.0          # exact fp16 midpoints (ties to even)
    edge = np.array([65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -26,
                     3 * 2.0 ** -26, 0.0, -0.0, 2.0 ** -14 - 2.0 ** -26])
    vals = np.concatenate([rand, mids, -mids, edge])
    ref = vals.astype(np.float16).view(np.uint16)
    got = oracle_lib.f64_to_f16(vals)
    assert np.array_equal(got, ref)


def test_bf16_round_matches_torch(oracle_lib):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    v32 = (rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000)).astype(np.float32)
    # fp32 values sitting exactly halfway between two bf16 values
    ties = ((rng.integers(0, 2**15, 2000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    v32 = np.concatenate([v32, ties[np.isfinite(ties)]])
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_lib.f64_to_bf16(v32.astype(np.float64))
    assert np.array_equal(got, ref)
    back = oracle_lib.bf16_to_f64(ref)
    tb = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    fin = np.isfinite(tb)
    assert np.array_equal(back[fin], tb[fin])


# ----------------------------------------------------------------------------
# unpackers: hand-enumerated cases

def test_sign1_hand_case(oracle_lib):
    g = _load("sign1_g128_hand.json")
    bits = _hex_array(g["bits_words_per_column"], np.uint32)
    scales = _hex_array(g["scales_f16_per_column"], np.uint16)
    W = oracle_lib.unpack(oracle_lib.FMT_SIGN1_G128, (bits, scales), g["K"], g["N"])
    for e in g["expected"]:
        assert W[e["k"], e["n"]] == e["w"], e
    # every weight is exactly +-s of its group (0 -> -s, 1 -> +s)
    s = np.abs(oracle_lib.f16_to_f64(scales))
    for n in range(g["N"]):
        for k in range(g["K"]):
            assert abs(W[k, n]) == s[n, k // 128]


def test_affine2_hand_case(oracle_lib):
    g = _load("affine2_hand.json")
    codes = _hex_array(g["codes_words_per_column"], np.uint32)
    scales = _hex_array(g["scales_f16_per_column"], np.uint16)
    biases = _hex_array(g["biases_f16_per_column"], np.uint16)
    W = oracle_lib.unpack(oracle_lib.FMT_AFFINE2, (codes, scales, biases), g["K"], g["N"],
                          g["group"])
    for e in g["expected"]:
        assert W[e["k"], e["n"]] == e["w"], e


def test_q4_0_hand_case(oracle_lib):
    g = _load("q4_0_hand.json")
    N, K = g["N"], g["K"]
    blocks = np.zeros((N, K // 32, 18), np.uint8)
    for n, col in enumerate(g["blocks_per_column"]):
        for b, blk in enumerate(col):
            d = int(blk["d_f16"], 16)
            blocks[n, b, 0] = d & 0xFF
            blocks[n, b, 1] = d >> 8
            blocks[n, b, 2:] = [int(v, 16) for v in blk["qs"]]
    W = oracle_lib.unpack(oracle_lib.FMT_Q4_0, (blocks,), K, N)
    for e in g["expected"]:
        assert W[e["k"], e["n"]] == e["w"], e


def test_affine2_unit_scale_gives_codes(oracle_lib):
    """scale 1, bias 0: w equals the 2-bit code itself; the codes of word
    0xE4E4E4E4 read 0,1,2,3 repeating (little end first)."""
    K, N = 64, 2
    codes = np.full((N, K // 16), 0xE4E4E4E4, np.uint32)
    one = np.full((N, 1), 0x3C00, np.uint16)
    zero = np.zeros((N, 1), np.uint16)
    W = oracle_lib.unpack(oracle_lib.FMT_AFFINE2, (codes, one, zero), K, N, 64)
    assert np.array_equal(W[:, 0], np.tile([0.0, 1.0, 2.0, 3.0], 16))


def test_size_identities():
    """Canonical byte counts: 1.125, 2 + 32/g and 4.5 bits per weight."""
    K, N = 5120, 256
    mat = synth.Matrix("w", synth.SIGN1_G128, K, N, 128, "f16")
    (bits, scales), _ = synth.gen_matrix(mat, 0, rows=1)
    assert Fraction((bits.nbytes + scales.nbytes) * 8, K * N) == Fraction(9, 8)
    for g, bpw in ((64, Fraction(5, 2)), (128, Fraction(9, 4))):
        mat = synth.Matrix("w", synth.AFFINE2, K, N, g, "f16")
        (c, s, b), _ = synth.gen_matrix(mat, 0, rows=1)
        assert Fraction((c.nbytes + s.nbytes + b.nbytes) * 8, K * N) == bpw
    mat = synth.Matrix("w", synth.Q4_0, K, N, 32, "f16")
    (blk,), _ = synth.gen_matrix(mat, 0, rows=1)
    assert Fraction(blk.nbytes * 8, K * N) == Fraction(9, 2)


def sign1_as_affine(bits, scales, K, N):
    """The same sign weights in MLX affine form: code = bit, scale 2s, bias -s."""
    b = ((bits[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(N, K)
    codes = (b.reshape(N, K // 16, 16).astype(np.uint32) << (2 * np.arange(16, dtype=np.uint32)))
    codes = np.bitwise_or.reduce(codes, axis=2).astype(np.uint32)
    s16 = scales.view(np.float16)
    s2 = (s16.astype(np.float32) * 2).astype(np.float16)
    assert np.all(s2.astype(np.float64) == 2 * s16.astype(np.float64))   # exact
    return codes, s2.view(np.uint16), (-s16).view(np.uint16)


def test_sign1_equals_affine_2s_minus_s(oracle_lib):
    """Bonsai-27B-mlx-1bit model card: the same sign weights stored in MLX's
    affine form use scale 2s and bias -s with q in {0,1}; that reproduces +-s
    exactly, so dequant and the verify product must be identical."""
    K, N, M = 512, 48, 5
    mat = synth.Matrix("w", synth.SIGN1_G128, K, N, 128, "f16")
    (bits, scales), xb = synth.gen_matrix(mat, 7, rows=M)
    aff = sign1_as_affine(bits, scales, K, N)
    W1 = oracle_lib.unpack(oracle_lib.FMT_SIGN1_G128, (bits, scales), K, N)
    W2 = oracle_lib.unpack(oracle_lib.FMT_AFFINE2, aff, K, N, 128)
    assert np.array_equal(W1, W2)
    X = oracle_lib.f16_to_f64(xb)
    Y1, _ = oracle_lib.verify(oracle_lib.FMT_SIGN1_G128, (bits, scales), X, K, N)
    Y2, _ = oracle_lib.verify(oracle_lib.FMT_AFFINE2, aff, X, K, N, 128)
    assert np.array_equal(Y1, Y2)
    D1 = oracle_lib.dequant_f16(oracle_lib.FMT_SIGN1_G128, (bits, scales), K, N)
    D2 = oracle_lib.dequant_f16(oracle_lib.FMT_AFFINE2, aff, K, N, 128)
    assert np.array_equal(D1, D2)


# ----------------------------------------------------------------------------
# dequant to fp16: round once from the exact value

def test_dequant_matches_numpy_rounding(oracle_lib):
    for mat in (synth.Matrix("w", synth.AFFINE2, 256, 32, 64, "f16", sigma_scale=0.01),
                synth.Matrix("w", synth.Q4_0, 256, 32, 32, "f16", sigma_scale=0.01),
                synth.Matrix("w", synth.SIGN1_G128, 256, 32, 128, "f16")):
        parts, _ = synth.gen_matrix(mat, 3, rows=1)
        W = oracle_lib.unpack(FMT[mat.fmt], parts, mat.K, mat.N, mat.group)
        D = oracle_lib.dequant_f16(FMT[mat.fmt], parts, mat.K, mat.N, mat.group)
        assert np.array_equal(D, W.astype(np.float16).view(np.uint16))
        cols = np.array([31, 2, 2])
        Dc = oracle_lib.dequant_f16(FMT[mat.fmt], parts, mat.K, mat.N, mat.group, cols=cols)
        assert np.array_equal(Dc, D[:, cols])


# ----------------------------------------------------------------------------
# the contraction

@pytest.mark.parametrize("fmtname", [synth.SIGN1_G128, synth.AFFINE2, synth.Q4_0])
def test_verify_equals_dense_and_numpy(oracle_lib, fmtname):
    """Packed = dense: the column-streamed verify equals the naive triple loop
    over the explicitly unpacked matrix bit for bit, and numpy's matmul within
    fp64 rounding."""
    K, N, M = 384, 40, 8
    group = {synth.SIGN1_G128: 128, synth.AFFINE2: 64, synth.Q4_0: 32}[fmtname]
    if fmtname == synth.SIGN1_G128:
        K = 512
    mat = synth.Matrix("w", fmtname, K, N, group, "f16", sigma_scale=0.01)
    parts, xb = synth.gen_matrix(mat, 11, rows=M)
    X = oracle_lib.f16_to_f64(xb)
    W = oracle_lib.unpack(FMT[fmtname], parts, K, N, group)
    Yd = oracle_lib.gemm(X, W)
    Yv, A = oracle_lib.verify(FMT[fmtname], parts, X, K, N, group)
    assert np.array_equal(Yd, Yv)
    Yn = X @ W
    assert np.all(np.abs(Yv - Yn) <= 1e-12 * (np.abs(X) @ np.abs(W)))
    assert np.allclose(A, np.abs(X) @ np.abs(W), rtol=1e-12)


def test_verify_brute_force_exact(oracle_lib):
    """Brute force at K=128, N=16 in exact rational arithmetic."""
    K, N, M = 128, 16, 3
    mat = synth.Matrix("w", synth.SIGN1_G128, K, N, 128, "f16")
    parts, xb = synth.gen_matrix(mat, 5, rows=M)
    X = oracle_lib.f16_to_f64(xb)
    W = oracle_lib.unpack(0, parts, K, N)
    Yv, A = oracle_lib.verify(0, parts, X, K, N)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(X[m, k])) * Fraction(float(W[k, n])) for k in range(K))
            # products x*w are exact in fp64; K additions add at most K half-ulps of A
            bound = Fraction(float(A[m, n])) * K * Fraction(1, 2**53)
            assert abs(Fraction(float(Yv[m, n])) - exact) <= bound


def test_verify_row_independence(oracle_lib):
    """An M-row result equals M single-row results (bit for bit)."""
    K, N, M = 256, 24, 8
    mat = synth.Matrix("w", synth.AFFINE2, K, N, 128, "bf16", sigma_scale=0.01)
    parts, xb = synth.gen_matrix(mat, 9, rows=M)
    X = oracle_lib.bf16_to_f64(xb)
    Y, _ = oracle_lib.verify(1, parts, X, K, N, 128)
    for m in range(M):
        Ym, _ = oracle_lib.verify(1, parts, X[m:m + 1], K, N, 128)
        assert np.array_equal(Ym[0], Y[m])


def test_verify_column_subset(oracle_lib):
    K, N = 256, 64
    mat = synth.Matrix("w", synth.Q4_0, K, N, 32, "f16", sigma_scale=0.01)
    parts, xb = synth.gen_matrix(mat, 4, rows=2)
    X = oracle_lib.f16_to_f64(xb)
    Y, _ = oracle_lib.verify(2, parts, X, K, N, 32)
    cols = np.array([63, 0, 17, 17, 40])
    Ys, _ = oracle_lib.verify(2, parts, X, K, N, 32, cols=cols)
    assert np.array_equal(Ys, Y[:, cols])


# ----------------------------------------------------------------------------
# the blockwise Hadamard rotation

def test_fwht_matches_scipy_sylvester(oracle_lib):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(128).astype(np.float64)     # Sylvester, natural order
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 384)).astype(np.float16).astype(np.float64)
    got = oracle_lib.fwht128(x)
    ref = np.concatenate([x[:, b * 128:(b + 1) * 128] @ H for b in range(3)], axis=1) / np.sqrt(128)
    assert np.allclose(got, ref, rtol=1e-15, atol=1e-15)


def test_fwht_closed_forms(oracle_lib):
    e0 = np.zeros(128)
    e0[0] = 1.0
    assert np.allclose(oracle_lib.fwht128(e0), np.full(128, 1 / np.sqrt(128)), rtol=1e-15)
    # the all-ones block maps to sqrt(128) e_0
    y = oracle_lib.fwht128(np.ones(128))
    assert abs(y[0] - np.sqrt(128)) < 1e-12 and np.max(np.abs(y[1:])) < 1e-12
    # Sylvester recursion H_2n = [[H_n, H_n], [H_n, -H_n]]: for x = [a, 0] the
    # two halves of H x are equal; for x = [0, a] they are negatives.
    rng = np.random.default_rng(3)
    a = rng.standard_normal(64)
    y1 = oracle_lib.fwht128(np.concatenate([a, np.zeros(64)]))
    y2 = oracle_lib.fwht128(np.concatenate([np.zeros(64), a]))
    assert np.allclose(y1[:64], y1[64:], rtol=0, atol=1e-13)
    assert np.allclose(y2[:64], -y2[64:], rtol=0, atol=1e-13)
    assert np.allclose(y1[:64], y2[:64], rtol=0, atol=1e-13)


def test_fwht_involution_and_parseval(oracle_lib):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 512))
    y = oracle_lib.fwht128(x)
    assert np.allclose(oracle_lib.fwht128(y), x, rtol=0, atol=1e-12)
    for b in range(4):
        blk = slice(b * 128, (b + 1) * 128)
        assert np.allclose(np.sum(y[:, blk] ** 2, axis=1), np.sum(x[:, blk] ** 2, axis=1),
                           rtol=1e-12)


def test_fwht_signs(oracle_lib):
    rng = np.random.default_rng(5)
    x = rng.standard_normal(256)
    signs = synth.random_signs(6, 256)
    sbits = ((signs[:, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(-1)
    xs = np.where(sbits == 1, -x, x)
    assert np.array_equal(oracle_lib.fwht128(x, signs), oracle_lib.fwht128(xs))


def test_rotation_invariance(oracle_lib):
    """(x H) . (H^T W) = x . W with the normalized block rotation: a matrix
    quantized in the rotated basis sees the rotated activations."""
    rng = np.random.default_rng(6)
    K, N = 256, 8
    x = rng.standard_normal((2, K))
    W = rng.standard_normal((K, N))
    W_rot = oracle_lib.fwht128(W.T).T          # each column rotated blockwise (H symmetric)
    lhs = oracle_lib.gemm(oracle_lib.fwht128(x), W_rot)
    assert np.allclose(lhs, x @ W, rtol=1e-12, atol=1e-12)


def test_fwht_exact_sum_then_one_rounding(oracle_lib):
    """For fp16 inputs the block sum is exact in fp64; the only rounding is
    the IEEE division by sqrt(128): compare with exact rational sums."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(128)
    rng = np.random.default_rng(8)
    x = rng.standard_normal(128).astype(np.float16).astype(np.float64)
    y = oracle_lib.fwht128(x)
    for i in range(0, 128, 9):
        s = sum(Fraction(float(x[j])) * int(H[i, j]) for j in range(128))
        assert float(s) / np.sqrt(128.0) == y[i]


# ----------------------------------------------------------------------------
# Greedy argmax (fused head epilogue)

def test_argmax_rows_hand_cases(oracle_lib):
    """Hand-made rows: first of tied maxima, -0 equal to +0, negative rows,
    the first NaN, a single column."""
    nan, inf = float("nan"), float("inf")
    Y = [[1.0, 3.0, 3.0, 2.0],
         [-1.0, -0.0, 0.0, -2.0],
         [-5.0, -3.0, -4.0, -3.0],
         [1.0, nan, 5.0, nan],
         [-inf, -inf, -inf, -inf],
         [2.0, 1.0, inf, 0.5]]
    assert oracle_lib.argmax_rows(np.array(Y)).tolist() == [1, 1, 1, 1, 0, 2]
    assert oracle_lib.argmax_rows(np.array([[7.0]])).tolist() == [0]


def test_argmax_rows_brute_force(oracle_lib):
    """Against a pairwise-comparison definition on small random rows with
    many ties (values drawn from a handful of levels)."""
    rng = np.random.default_rng(11)
    Y = rng.integers(-3, 4, size=(50, 9)).astype(np.float64)
    got = oracle_lib.argmax_rows(Y)
    for m in range(Y.shape[0]):
        best = [n for n in range(9) if all(Y[m, n] >= Y[m, j] for j in range(9))]
        assert got[m] == best[0]
