"""CPU tests of the seeded input generators (synth): they are deterministic,
follow the documented draw order and canonical layouts, and their values have
the documented distributions; the workloads have the documented shapes."""
import numpy as np
import pytest

import synth

SHAPES = {
    synth.SIGN1_G128: lambda K, N, g: [(N, K // 32), (N, K // 128)],
    synth.AFFINE2: lambda K, N, g: [(N, K // 16), (N, K // g), (N, K // g)],
    synth.Q4_0: lambda K, N, g: [(N, K // 32, 18)],
}


def f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def bf16_rne(x32):
    """Round float32 to bf16 bits, nearest even, from the bit patterns."""
    u = np.asarray(x32, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("fmt,K,N,g,xd", [
    (synth.SIGN1_G128, 512, 96, 128, "f16"), (synth.AFFINE2, 384, 40, 64, "bf16"),
    (synth.AFFINE2, 256, 24, 32, "f16"), (synth.Q4_0, 320, 33, 32, "f16")])
def test_layouts_and_determinism(fmt, K, N, g, xd):
    mat = synth.Matrix("w", fmt, K, N, g, xd)
    parts, xb = synth.gen_matrix(mat, 5, rows=8)
    assert [p.shape for p in parts] == SHAPES[fmt](K, N, g)
    assert xb.shape == (8, K) and xb.dtype == np.uint16
    again, xb2 = synth.gen_matrix(mat, 5, rows=8)
    assert all(np.array_equal(a, b) for a, b in zip(parts, again)) and np.array_equal(xb, xb2)
    other, xb3 = synth.gen_matrix(mat, 6, rows=8)
    assert not np.array_equal(parts[0], other[0]) and not np.array_equal(xb, xb3)


def test_draw_order_sign1():
    """Codes, then scales, then X, from one PCG64 stream."""
    mat = synth.Matrix("w", synth.SIGN1_G128, 256, 16, 128, "f16")
    (bits, scales), xb = synth.gen_matrix(mat, 11, rows=3)
    rng = np.random.default_rng(11)
    assert np.array_equal(bits, rng.integers(0, 2**32, size=(16, 8), dtype=np.uint32))
    s = np.abs(rng.normal(0.0, 0.02, (16, 2)))
    assert np.array_equal(scales, s.astype(np.float16).view(np.uint16))
    x = rng.standard_normal((3, 256), dtype=np.float32)
    assert np.array_equal(xb, x.astype(np.float16).view(np.uint16))


def test_draw_order_affine2_bf16():
    """Codes, scales, biases, then X rounded to bf16 (nearest even)."""
    mat = synth.Matrix("w", synth.AFFINE2, 128, 8, 64, "bf16", sigma_scale=0.01)
    (codes, scales, biases), xb = synth.gen_matrix(mat, 3, rows=2)
    rng = np.random.default_rng(3)
    assert np.array_equal(codes, rng.integers(0, 2**32, size=(8, 8), dtype=np.uint32))
    assert np.array_equal(scales, np.abs(rng.normal(0.0, 0.01, (8, 2))).astype(np.float16)
                          .view(np.uint16))
    assert np.array_equal(biases, rng.normal(0.0, 0.01, (8, 2)).astype(np.float16)
                          .view(np.uint16))
    assert np.array_equal(xb, bf16_rne(rng.standard_normal((2, 128), dtype=np.float32)))


def test_distributions():
    K, N = 4096, 256
    (bits, scales), xb = synth.gen_matrix(synth.Matrix("w", synth.SIGN1_G128, K, N, 128, "f16"), 1)
    ones = np.unpackbits(bits.view(np.uint8)).mean()
    assert abs(ones - 0.5) < 0.005                         # signs Bernoulli(0.5)
    s = f16(scales)
    assert np.all(s >= 0) and np.all(np.isfinite(s))
    assert abs(np.median(s) / 0.02 - 0.6745) < 0.05        # |N(0, sigma)|: median 0.6745 sigma
    x = f16(xb)
    assert np.all(np.isfinite(x)) and abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02

    (codes, sc, bi), _ = synth.gen_matrix(synth.Matrix("w", synth.AFFINE2, K, N, 64, "f16"), 2)
    q = np.stack([(codes >> (2 * i)) & 3 for i in range(16)]).ravel()
    assert np.allclose(np.bincount(q, minlength=4) / q.size, 0.25, atol=0.003)
    b = f16(bi)
    assert abs(b.mean()) < 0.0005 and abs(b.std() / 0.01 - 1) < 0.03

    (blocks,), _ = synth.gen_matrix(synth.Matrix("w", synth.Q4_0, K, N, 32, "f16"), 3)
    nib = np.concatenate([(blocks[:, :, 2:] & 15).ravel(), (blocks[:, :, 2:] >> 4).ravel()])
    assert np.allclose(np.bincount(nib, minlength=16) / nib.size, 1 / 16, atol=0.002)
    d = f16(blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
    assert np.all(d >= 0) and np.all(np.isfinite(d))


def test_workload_shapes():
    W = synth.WORKLOADS
    assert [(m.fmt, m.K, m.N, m.group, m.xdtype) for m in W["sign1_tiny_512x256"].matrices] == \
        [(synth.SIGN1_G128, 512, 256, 128, "f16")]
    assert [(m.K, m.N, m.group, m.xdtype) for m in W["sign1_mlp_up_5120x17408"].matrices] == \
        [(5120, 17408, 128, "f16")]
    assert [(m.fmt, m.K, m.N, m.group, m.xdtype) for m in W["affine2_g64_6144x6144"].matrices] == \
        [(synth.AFFINE2, 6144, 6144, 64, "bf16")]
    assert [(m.K, m.N, m.group) for m in W["affine2_g64_kv_5120x1024"].matrices] == \
        [(5120, 1024, 64)]
    (head,) = W["head_rot_affine2_g128_5120x151936"].matrices
    assert (head.fmt, head.K, head.N, head.group, head.rotate) == \
        (synth.AFFINE2, 5120, 151936, 128, True)
    stack = W["q4_0_stack_4x7"].matrices
    assert len(stack) == 28 and all(m.fmt == synth.Q4_0 for m in stack)
    layer = [(m.K, m.N) for m in stack[:7]]
    assert layer == [(5120, 6144), (5120, 1024), (5120, 1024), (6144, 5120), (5120, 17408),
                     (5120, 17408), (17408, 5120)]
    assert sum(N * (K // 32) * 18 for K, N in layer) == 191692800     # bytes per layer


def test_matrix_seeds():
    single = synth.WORKLOADS["sign1_tiny_512x256"]
    assert synth.matrix_seed(single, 0) == single.seed
    stack = synth.WORKLOADS["q4_0_stack_4x7"]
    assert synth.matrix_seed(stack, 3) == [stack.seed, 3]
    a = synth.gen_matrix(synth.Matrix("w", synth.Q4_0, 64, 16, 32, "f16"), [0, 1])[0][0]
    b = synth.gen_matrix(synth.Matrix("w", synth.Q4_0, 64, 16, 32, "f16"), [0, 2])[0][0]
    assert not np.array_equal(a, b)
    signs = synth.random_signs(4, 256)
    assert signs.shape == (8,) and signs.dtype == np.uint32
