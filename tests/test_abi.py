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
    assert lbv.packed_bytes(lbv.FMT_SIGN1_G128, 384, 20) == 3 * 128 * (16 + 2)
    assert lbv.packed_bytes(lbv.FMT_AFFINE2, 96, 17, 32) == 2 * 128 * (16 + 8)
    assert lbv.packed_bytes(lbv.FMT_Q4_0, 96, 129, 32) == 2 * 2 * 128 * (32 + 4)


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
    h = P()
    assert L.lbv_plan_create(1, 128, 16, 48, 0, 0, ctypes.byref(h)) == lbv.ERR_UNSUPPORTED
    assert h.value is None
    assert L.lbv_plan_create(0, 100, 16, 128, 0, 0, ctypes.byref(h)) == lbv.ERR_INVALID_ARG
    assert L.lbv_plan_create(0, 128, 16, 128, 5, 0, ctypes.byref(h)) == lbv.ERR_INVALID_ARG
    assert L.lbv_plan_create(0, 128, 16, 128, 0, 0x6, ctypes.byref(h)) == lbv.ERR_INVALID_ARG


# ----------------------------------------------------------------------------
# The device layout, read back from its written specification (layout.h):
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


@pytest.mark.parametrize("fmt,K,N,group", [
    (lbv.FMT_SIGN1_G128, 512, 48, 128), (lbv.FMT_SIGN1_G128, 384, 150, 128),
    (lbv.FMT_AFFINE2, 256, 32, 64), (lbv.FMT_AFFINE2, 320, 17, 32), (lbv.FMT_AFFINE2, 384, 140, 128),
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
    ck = SPEC[fmt][group][0]
    gk = group if fmt == lbv.FMT_AFFINE2 else (128 if fmt == lbv.FMT_SIGN1_G128 else 32)
    per = 2 if fmt == lbv.FMT_AFFINE2 else 1          # fp16 values per group
    ntiles, nch = side.shape[0], side.shape[1]
    for tile in range(ntiles):
        for ch in range(nch):
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
