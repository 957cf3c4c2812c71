"""Seeded synthetic inputs for the few-row packed-weight verify matmul.

This module only draws random numbers and lays them out in the canonical
(file) layouts; it holds none of the method's arithmetic.  Both the CPU oracle
and the CUDA library consume exactly the arrays produced here.

Draw order for one matrix, from ``numpy.random.default_rng(seed)`` (PCG64):
  1. codes (sign bits / 2-bit codes / Q4_0 nibbles), as uniform uint32 or
     uint8 words: every bit (or code) is independent and uniform, i.e. signs are
     Bernoulli(0.5), 2-bit q uniform in {0..3}, 4-bit q uniform in {0..15};
  2. scales (or Q4_0 d): |N(0, sigma)| rounded to fp16;
  3. biases (affine only): N(0, 0.01) rounded to fp16;
  4. X [8, K]: N(0, 1) drawn as float32, rounded to fp16 or bf16 (RNE).
A call with M rows uses the first M rows of X.

Canonical layouts:
  sign1 g128: bits uint32 [N, K/32] (bit k%32 of word k/32), scales uint16 [N, K/128]
  affine2 g:  codes uint32 [N, K/16] (2 bits per code, little end first),
              scales uint16 [N, K/g], biases uint16 [N, K/g]
  q4_0:       blocks uint8 [N, K/32, 18] = {d (fp16 LE), qs[16]}
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SIGN1_G128 = "sign1_g128"
AFFINE2 = "affine2"
Q4_0 = "q4_0"


@dataclass(frozen=True)
class Matrix:
    """One packed weight matrix of a workload."""
    name: str
    fmt: str
    K: int
    N: int
    group: int          # 128 for sign1, the affine group, 32 for Q4_0
    xdtype: str         # "f16" or "bf16"
    rotate: bool = False  # activations rotated blockwise by H128/sqrt(128)
    sigma_scale: float = 0.02
    sigma_bias: float = 0.01


@dataclass(frozen=True)
class Workload:
    name: str
    matrices: tuple = field(default_factory=tuple)
    seed: int = 0


def _q4_stack():
    shapes = [("q", 5120, 6144), ("k", 5120, 1024), ("v", 5120, 1024), ("o", 6144, 5120),
              ("gate", 5120, 17408), ("up", 5120, 17408), ("down", 17408, 5120)]
    mats = []
    for layer in range(4):
        for nm, K, N in shapes:
            mats.append(Matrix(f"l{layer}.{nm}", Q4_0, K, N, 32, "f16", sigma_scale=0.01))
    return tuple(mats)


WORKLOADS = {
    # 1-bit sign g128, K=512, N=256, fp16 rows, seed 0 (the tiny parity case)
    "sign1_tiny_512x256": Workload("sign1_tiny_512x256",
                                   (Matrix("w", SIGN1_G128, 512, 256, 128, "f16"),)),
    # 1-bit sign g128 MLP-up projection
    "sign1_mlp_up_5120x17408": Workload("sign1_mlp_up_5120x17408",
                                        (Matrix("up", SIGN1_G128, 5120, 17408, 128, "f16"),)),
    # 2-bit affine g64 with bf16 rows: a 6144-wide projection and an attention k/v
    "affine2_g64_6144x6144": Workload("affine2_g64_6144x6144",
                                      (Matrix("proj", AFFINE2, 6144, 6144, 64, "bf16",
                                              sigma_scale=0.01),)),
    "affine2_g64_kv_5120x1024": Workload("affine2_g64_kv_5120x1024",
                                         (Matrix("kv", AFFINE2, 5120, 1024, 64, "bf16",
                                                 sigma_scale=0.01),)),
    # Hadamard-rotated 2-bit g128 output head
    "head_rot_affine2_g128_5120x151936": Workload(
        "head_rot_affine2_g128_5120x151936",
        (Matrix("head", AFFINE2, 5120, 151936, 128, "f16", rotate=True, sigma_scale=0.01),)),
    # GGUF Q4_0 layer stack, 4 layers x {q, k, v, o, gate, up, down}
    "q4_0_stack_4x7": Workload("q4_0_stack_4x7", _q4_stack()),
}


def _f16_bits(a) -> np.ndarray:
    return np.asarray(a).astype(np.float16).view(np.uint16)


def _bf16_bits(a32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def x_bits(rng, M: int, K: int, xdtype: str) -> np.ndarray:
    x = rng.standard_normal((M, K), dtype=np.float32)
    return _f16_bits(x) if xdtype == "f16" else _bf16_bits(x)


def gen_matrix(mat: Matrix, seed, rows: int = 8):
    """Returns (parts, xbits): the canonical packed arrays and X bits [rows, K]."""
    rng = np.random.default_rng(seed)
    K, N, g = mat.K, mat.N, mat.group
    if mat.fmt == SIGN1_G128:
        assert K % 128 == 0
        bits = rng.integers(0, 2**32, size=(N, K // 32), dtype=np.uint32)
        scales = _f16_bits(np.abs(rng.normal(0.0, mat.sigma_scale, (N, K // 128))))
        parts = (bits, scales)
    elif mat.fmt == AFFINE2:
        assert K % 16 == 0 and K % g == 0
        codes = rng.integers(0, 2**32, size=(N, K // 16), dtype=np.uint32)
        scales = _f16_bits(np.abs(rng.normal(0.0, mat.sigma_scale, (N, K // g))))
        biases = _f16_bits(rng.normal(0.0, mat.sigma_bias, (N, K // g)))
        parts = (codes, scales, biases)
    elif mat.fmt == Q4_0:
        assert K % 32 == 0
        qs = rng.integers(0, 256, size=(N, K // 32, 16), dtype=np.uint8)
        d = _f16_bits(np.abs(rng.normal(0.0, mat.sigma_scale, (N, K // 32))))
        blocks = np.empty((N, K // 32, 18), np.uint8)
        blocks[:, :, 0] = (d & 0xFF).astype(np.uint8)
        blocks[:, :, 1] = (d >> 8).astype(np.uint8)
        blocks[:, :, 2:] = qs
        parts = (blocks,)
    else:
        raise ValueError(mat.fmt)
    xb = x_bits(rng, rows, K, mat.xdtype)
    return parts, xb


def matrix_seed(workload: Workload, index: int):
    """Seed of the index-th matrix of a workload (a single matrix uses the bare seed)."""
    if len(workload.matrices) == 1:
        return workload.seed
    return [workload.seed, index]


def gen_workload(name: str, seed: int | None = None, rows: int = 8):
    wl = WORKLOADS[name]
    if seed is not None:
        wl = Workload(wl.name, wl.matrices, seed)
    out = []
    for i, mat in enumerate(wl.matrices):
        parts, xb = gen_matrix(mat, matrix_seed(wl, i), rows)
        out.append((mat, parts, xb))
    return out


def random_signs(seed, K: int) -> np.ndarray:
    """A random +-1 diagonal for the randomized rotation: K bits as uint32 [K/32]."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 2**32, size=(K // 32,), dtype=np.uint32)
