"""CPU tests of the C ABI: the library builds and loads, exports every entry
point include/lbv.h declares, rejects bad arguments with status codes, and its
host packers are lossless rearrangements of the canonical layouts."""
import ctypes
import os
import re

import numpy as np
import pytest

import few_row_packed_gb300 as lbv
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lbv.h")


@pytest.fixture(scope="module")
def L():
    lbv.build()
    return lbv.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^LBV_API [^(]*?\b(lbv_\w+)\(", text, re.M)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    out = os.popen(f"nm -D --defined-only {lbv.LIB_PATH}").read()
    exported = set(re.findall(r" T (lbv_\w+)", out))
    assert set(names) == exported, (set(names) ^ exported)


def test_version(L):
    assert "sm_103a" in lbv.version()


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(lbv, "_lib", None)
    monkeypatch.setattr(lbv, "LIB_PATH", "/nonexistent/liblbv.so")
    with pytest.raises(RuntimeError, match="missing"):
        lbv.lib()


def test_packed_bytes_identities(L):
    assert lbv.packed_bytes(lbv.FMT_SIGN1_G128, 5120, 17408) == 5120 * 17408 * 9 // 64
    assert lbv.packed_bytes(lbv.FMT_AFFINE2, 6144, 6144, 64) == 6144 * 6144 * 5 // 16
    assert lbv.packed_bytes(lbv.FMT_AFFINE2, 5120, 1024, 64) == 5120 * 1024 * 5 // 16
    assert lbv.packed_bytes(lbv.FMT_AFFINE2, 5120, 151936, 128) == 218787840
    assert lbv.packed_bytes(lbv.FMT_Q4_0, 5120, 17408, 32) == 5120 * 17408 * 9 // 16
    q4 = sum(lbv.packed_bytes(lbv.FMT_Q4_0, K, N, 32) for _, K, N in
             [("q", 5120, 6144), ("k", 5120, 1024), ("v", 5120, 1024), ("o", 6144, 5120),
              ("g", 5120, 17408), ("u", 5120, 17408), ("d", 17408, 5120)])
    assert q4 == 191692800
    # invalid shapes
    assert lbv.packed_bytes(lbv.FMT_SIGN1_G128, 100, 16) == 0
    assert lbv.packed_bytes(lbv.FMT_SIGN1_G128, 128, 0) == 0
    assert lbv.packed_bytes(lbv.FMT_AFFINE2, 128, 16, 48) == 0
    assert lbv.packed_bytes(lbv.FMT_Q4_0, 48, 16, 32) == 0
    assert lbv.packed_bytes(7, 128, 16, 128) == 0
    # padding: ragged N and K round up to a tile and a chunk
    assert lbv.packed_bytes(lbv.FMT_SIGN1_G128, 384, 20) == 2 * 2 * (512 + 8 * 8)
    assert lbv.packed_bytes(lbv.FMT_AFFINE2, 96, 17, 32) == 2 * 1 * (512 + 8 * 32)


def test_bad_arguments_return_status(L):
    P = ctypes.c_void_p
    assert L.lbv_verify_gemm(None, None, 1, 1, None, None, 1, None, 0, None) == lbv.ERR_INVALID_ARG
    assert "plan" in lbv.last_error()
    assert L.lbv_plan_query(None, 1, None, None, None) == lbv.ERR_INVALID_ARG
    assert L.lbv_pack_sign_g128(None, None, 128, 16, None, 0) == lbv.ERR_INVALID_ARG
    buf = np.zeros(16, np.uint8)
    bits = np.zeros(4 * 16, np.uint32)
    sc = np.zeros(16, np.uint16)
    st = L.lbv_pack_sign_g128(bits.ctypes.data, sc.ctypes.data, 128, 16, buf.ctypes.data, buf.size)
    assert st == lbv.ERR_WORKSPACE
    assert L.lbv_fwht128(None, None, 1, 128, 0, None, None) == lbv.ERR_INVALID_ARG
    x = np.zeros(256, np.uint16)
    assert L.lbv_fwht128(x.ctypes.data, x.ctypes.data, 1, 100, 0, None, None) == lbv.ERR_INVALID_ARG
    assert L.lbv_fwht128(x.ctypes.data, x.ctypes.data, 9, 128, 0, None, None) == lbv.ERR_INVALID_ARG
    assert L.lbv_fused_rotation(None, None, 1, 128, 0, None, None) == lbv.ERR_INVALID_ARG
    assert L.lbv_fused_rotation(x.ctypes.data, x.ctypes.data, 1, 96, 0, None, None) == \
        lbv.ERR_INVALID_ARG
    assert L.lbv_fused_rotation(x.ctypes.data, x.ctypes.data, 0, 128, 0, None, None) == \
        lbv.ERR_INVALID_ARG
    assert L.lbv_verify_fused(None, None, 1, 1, None, lbv.FUSED_ARGMAX, None, None, 1, None,
                              None, None, 0, None) == lbv.ERR_INVALID_ARG
    assert "lbv_verify_fused" in lbv.last_error()
    assert lbv.fused_workspace_bytes() == 128
    K = (ctypes.c_int * 2)(128, 128)
    N = (ctypes.c_int * 2)(16, 16)
    assert L.lbv_group_create(2, 32, 0, 0, K, N, 0, ctypes.byref(P())) == lbv.ERR_INVALID_ARG
    assert L.lbv_group_create(2, 32, 0, 2, K, N, 0x2, ctypes.byref(P())) == lbv.ERR_INVALID_ARG
    K[1] = 100
    assert L.lbv_group_create(2, 32, 0, 2, K, N, 0, ctypes.byref(P())) == lbv.ERR_INVALID_ARG
    assert "problem 1" in lbv.last_error()
    assert L.lbv_verify_grouped(None, None, None) == lbv.ERR_INVALID_ARG
    assert ctypes.sizeof(lbv.Problem) == 40
    h = P()
    assert L.lbv_plan_create(1, 128, 16, 48, 0, 0, ctypes.byref(h)) == lbv.ERR_UNSUPPORTED
    assert h.value is None
    assert L.lbv_plan_create(0, 100, 16, 128, 0, 0, ctypes.byref(h)) == lbv.ERR_INVALID_ARG
    assert L.lbv_plan_create(0, 128, 16, 128, 5, 0, ctypes.byref(h)) == lbv.ERR_INVALID_ARG
    assert L.lbv_plan_create(0, 128, 16, 128, 0, 0x6, ctypes.byref(h)) == lbv.ERR_INVALID_ARG


# ----------------------------------------------------------------------------
# The device layout, read back from its written specification (layout.h):
# one record per (tile, chunk) in tile-major order, 512 code bytes
# [lane][word] then 8 x SB side bytes [g].  Word wi of lane (g, t) is column
# 16*tile + g + 8*(wi & 1), k-tiles (wi >> 1)*KT/2 + s//2; slot s holds the
# codes of k0 = 16*kt + 8*(s & 1) + 2*t at bit s*W and of k0+1 at 16 + s*W.

SPEC = {  # chunk_k, W (bits), slots
    lbv.FMT_SIGN1_G128: (256, 1, 16),
    lbv.FMT_AFFINE2: (128, 2, 8),
    lbv.FMT_Q4_0: (64, 4, 4),
}


def side_bytes(fmt, group):
    return (128 // group) * 8 if fmt == lbv.FMT_AFFINE2 else 8


def read_layout(fmt, packed, K, N, group):
    ck, W, slots = SPEC[fmt]
    KT = ck // 16
    ntiles, nch = -(-N // 16), -(-K // ck)
    rec = 512 + 8 * side_bytes(fmt, group)
    recs = packed.reshape(ntiles, nch, rec)
    codes = np.ascontiguousarray(recs[:, :, :512]).view(np.uint32).reshape(ntiles, nch, 32, 4)
    out = np.full((ntiles * 16, nch * ck), -1, np.int64)
    mask = (1 << W) - 1
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        for wi in range(4):
            n = np.arange(ntiles) * 16 + g + 8 * (wi & 1)
            for s in range(slots):
                kt = (wi >> 1) * (KT // 2) + (s >> 1)
                for h in range(2):
                    k = np.arange(nch) * ck + 16 * kt + 8 * (s & 1) + 2 * t + h
                    v = (codes[:, :, lane, wi] >> np.uint32(s * W + 16 * h)) & mask
                    out[np.ix_(n, k)] = v
    side = np.ascontiguousarray(recs[:, :, 512:]).view(np.uint16).reshape(ntiles, nch, 8, -1)
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


@pytest.mark.parametrize("fmt,K,N,group", [
    (lbv.FMT_SIGN1_G128, 512, 48, 128), (lbv.FMT_SIGN1_G128, 384, 21, 128),
    (lbv.FMT_AFFINE2, 256, 32, 64), (lbv.FMT_AFFINE2, 320, 17, 32), (lbv.FMT_AFFINE2, 384, 40, 128),
    (lbv.FMT_Q4_0, 192, 32, 32), (lbv.FMT_Q4_0, 96, 9, 32)])
def test_pack_is_lossless(L, fmt, K, N, group):
    name = {0: synth.SIGN1_G128, 1: synth.AFFINE2, 2: synth.Q4_0}[fmt]
    mat = synth.Matrix("w", name, K, N, group, "f16")
    parts, _ = synth.gen_matrix(mat, 13, rows=1)
    packed = lbv.pack(fmt, parts, K, N, group)
    assert packed.size == lbv.packed_bytes(fmt, K, N, group)
    codes, side = read_layout(fmt, packed, K, N, group)
    ref = canonical_codes(fmt, parts, K, N)
    assert np.array_equal(codes[:N, :K], ref)
    assert np.all(codes[N:, :] == 0) and np.all(codes[:, K:] == 0)
    ck = SPEC[fmt][0]
    # side entries: per group j of a chunk: scale(g), scale(g+8) [, bias(g), bias(g+8)]
    gk = group if fmt == lbv.FMT_AFFINE2 else (128 if fmt == lbv.FMT_SIGN1_G128 else 32)
    per = 4 if fmt == lbv.FMT_AFFINE2 else 2
    ntiles = side.shape[0]
    for tile in range(ntiles):
        for ch in range(side.shape[1]):
            for g in range(8):
                for j in range(ck // gk):
                    grp = ch * (ck // gk) + j
                    for hi in range(2):
                        n = tile * 16 + g + 8 * hi
                        e = side[tile, ch, g, per * j + hi]
                        if n >= N or grp * gk >= K:
                            assert e == 0
                        elif fmt == lbv.FMT_Q4_0:
                            blk = parts[0][n, grp]
                            assert e == int(blk[0]) | (int(blk[1]) << 8)
                        else:
                            assert e == parts[1][n, grp]
                            if fmt == lbv.FMT_AFFINE2:
                                assert side[tile, ch, g, per * j + 2 + hi] == parts[2][n, grp]
