"""Seeded synthetic inputs for the 4-bit GEMV (shared by tests, bench, smoke).

This module only draws random field values and places them at their byte
offsets; it holds none of the method's arithmetic (no dequantization, no
product).  Both the CUDA path and the CPU oracle consume what it produces.

Field distributions (the workloads of the skinny GEMV study):
  * Q4_K / Q5_K: d and dmin fp16 |N(0, 0.01)|, 12 packed 6-bit scale/min
    bytes uniform, qs (and Q5_K qh) bytes uniform.
  * Q6_K: ql, qh bytes uniform, int8 scales clip(round(N(0, 32))), d as above.
  * NVFP4: e2m1 code bytes uniform (all 16 codes), e4m3 group scales uniform
    over the 81 codes whose values lie in [2^-6, 16], one fp32 per-tensor
    scale uniform in [0.5, 1).
  * FP8 (block-scaled e4m3, one bf16 scale per 128 x 128 block): codes
    uniform over the 254 finite e4m3 codes (0x7F and 0xFF, the NaNs,
    excluded); scales bf16(2^u) with u uniform in [-10, -6] (the size of a
    block maximum over 448 for weights of a few hundredths).
  * x and residual: fp16 N(0, 1), rounded to nearest.

Every tensor has its own stream: numpy's SeedSequence keyed by
(seed, stream id), or a torch CUDA generator seeded from the same pair for
the multi-gigabyte bench sets.
"""
from __future__ import annotations

import numpy as np

Q4_K = 12
Q5_K = 13
Q6_K = 14
NVFP4 = 256
FP8 = 257

BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210}
TYPE_NAMES = {Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K", NVFP4: "NVFP4", FP8: "FP8"}

# e4m3 codes 0x08 (2^-6, the smallest normal) .. 0x58 (16): 81 codes.
E4M3_CODE_LO = 0x08
E4M3_CODE_HI = 0x58


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(stream)]))


def row_bytes(qtype: int, K: int) -> int:
    if qtype == NVFP4:
        return K // 2
    if qtype == FP8:
        return K
    return (K // 256) * BLOCK_BYTES[qtype]


def _abs_normal_f16(rng, shape, sigma=0.01) -> np.ndarray:
    return np.abs(rng.normal(0.0, sigma, size=shape)).astype(np.float16)


def q4k_weights(M: int, K: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Packed Q4_K matrix, uint8 [M][K/256*144]."""
    rng = _rng(seed, stream)
    nb = K // 256
    blk = np.empty((M, nb, 144), dtype=np.uint8)
    blk[..., 0:2] = _abs_normal_f16(rng, (M, nb)).view(np.uint8).reshape(M, nb, 2)
    blk[..., 2:4] = _abs_normal_f16(rng, (M, nb)).view(np.uint8).reshape(M, nb, 2)
    blk[..., 4:144] = rng.integers(0, 256, size=(M, nb, 140), dtype=np.uint8)
    return blk.reshape(M, nb * 144)


def q5k_weights(M: int, K: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Packed Q5_K matrix, uint8 [M][K/256*176]."""
    rng = _rng(seed, stream)
    nb = K // 256
    blk = np.empty((M, nb, 176), dtype=np.uint8)
    blk[..., 0:2] = _abs_normal_f16(rng, (M, nb)).view(np.uint8).reshape(M, nb, 2)
    blk[..., 2:4] = _abs_normal_f16(rng, (M, nb)).view(np.uint8).reshape(M, nb, 2)
    blk[..., 4:176] = rng.integers(0, 256, size=(M, nb, 172), dtype=np.uint8)
    return blk.reshape(M, nb * 176)


def q6k_weights(M: int, K: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Packed Q6_K matrix, uint8 [M][K/256*210]."""
    rng = _rng(seed, stream)
    nb = K // 256
    blk = np.empty((M, nb, 210), dtype=np.uint8)
    blk[..., 0:192] = rng.integers(0, 256, size=(M, nb, 192), dtype=np.uint8)
    sc = np.clip(np.rint(rng.normal(0.0, 32.0, size=(M, nb, 16))), -128, 127).astype(np.int8)
    blk[..., 192:208] = sc.view(np.uint8)
    blk[..., 208:210] = _abs_normal_f16(rng, (M, nb)).view(np.uint8).reshape(M, nb, 2)
    return blk.reshape(M, nb * 210)


def nvfp4_weights(M: int, K: int, seed: int = 0, stream: int = 0):
    """(codes uint8 [M][K/2], e4m3 scales uint8 [M][K/16], global scale)."""
    rng = _rng(seed, stream)
    codes = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    scales = rng.integers(E4M3_CODE_LO, E4M3_CODE_HI + 1, size=(M, K // 16), dtype=np.uint8)
    g = float(np.float32(rng.uniform(0.5, 1.0)))
    return codes, scales, g


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    """float32 values -> bf16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def fp8_weights(M: int, K: int, seed: int = 0, stream: int = 0):
    """(codes uint8 [M][K], bf16 scales as uint16 bits [ceil(M/128)][K/128], 1.0)."""
    rng = _rng(seed, stream)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    codes = finite[rng.integers(0, finite.size, size=(M, K))]
    u = rng.uniform(-10.0, -6.0, size=((M + 127) // 128, K // 128))
    scales = _bf16_bits(np.exp2(u).astype(np.float32))
    return codes, scales, 1.0


def weights(qtype: int, M: int, K: int, seed: int = 0, stream: int = 0):
    """(packed bytes, scales or None, global scale) for any supported type."""
    if qtype == Q4_K:
        return q4k_weights(M, K, seed, stream), None, 1.0
    if qtype == Q5_K:
        return q5k_weights(M, K, seed, stream), None, 1.0
    if qtype == Q6_K:
        return q6k_weights(M, K, seed, stream), None, 1.0
    if qtype == NVFP4:
        return nvfp4_weights(M, K, seed, stream)
    if qtype == FP8:
        return fp8_weights(M, K, seed, stream)
    raise ValueError(f"unknown type {qtype}")


def activations(N: int, K: int, seed: int = 0, stream: int = 1000,
                duplicate_rows: bool = False) -> np.ndarray:
    """fp16 x [N][K] ~ N(0, 1).  With duplicate_rows, every row t with
    t % 3 == 2 repeats row t - 2 (rows that share inputs)."""
    rng = _rng(seed, stream)
    x = rng.normal(0.0, 1.0, size=(N, K)).astype(np.float16)
    if duplicate_rows:
        for t in range(2, N, 3):
            x[t] = x[t - 2]
    return x


def residual(N: int, M: int, seed: int = 0, stream: int = 2000) -> np.ndarray:
    rng = _rng(seed, stream)
    return rng.normal(0.0, 1.0, size=(N, M)).astype(np.float16)


# ---------------------------------------------------------------------------
# Device-side generation for the multi-gigabyte bench sets (torch CUDA RNG).
# Same distributions; a different (but seeded) bit stream than the host path.
# ---------------------------------------------------------------------------

def _torch_gen(seed: int, stream: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(stream)) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def device_weights(qtype: int, M: int, K: int, seed: int, stream: int, device="cuda"):
    """Packed weights generated on the device: (bytes uint8 [M][row_bytes],
    scales uint8 [M][K/16] or None, global scale)."""
    import torch
    gen = _torch_gen(seed, stream, device)
    if qtype == FP8:
        codes = torch.randint(0, 254, (M, K), generator=gen, device=device, dtype=torch.int16)
        # 0..253 -> the 254 finite codes (skip 0x7F)
        codes = torch.where(codes >= 0x7F, codes + 1, codes).to(torch.uint8)
        u = torch.rand(((M + 127) // 128, K // 128), generator=gen, device=device) * 4.0 - 10.0
        scales = torch.exp2(u).to(torch.bfloat16).view(torch.int16).view(torch.uint8)
        return codes, scales.reshape((M + 127) // 128, 2 * (K // 128)), 1.0
    if qtype == NVFP4:
        codes = torch.randint(0, 256, (M, K // 2), generator=gen, device=device,
                              dtype=torch.uint8)
        scales = torch.randint(E4M3_CODE_LO, E4M3_CODE_HI + 1, (M, K // 16), generator=gen,
                               device=device, dtype=torch.uint8)
        gsc = float(np.float32(0.5 + 0.5 * torch.rand((), generator=gen, device=device).item()))
        return codes, scales, gsc
    bb = BLOCK_BYTES[qtype]
    nb = K // 256
    blk = torch.randint(0, 256, (M, nb, bb), generator=gen, device=device, dtype=torch.uint8)

    def f16_field():
        v = (torch.randn((M, nb), generator=gen, device=device) * 0.01).abs().half()
        return v.view(torch.uint8).view(M, nb, 2)

    if qtype in (Q4_K, Q5_K):
        blk[..., 0:2] = f16_field()
        blk[..., 2:4] = f16_field()
    else:
        sc = torch.randn((M, nb, 16), generator=gen, device=device) * 32.0
        sc = sc.round().clamp(-128, 127).to(torch.int8)
        blk[..., 192:208] = sc.view(torch.uint8)
        blk[..., 208:210] = f16_field()
    return blk.view(M, nb * bb), None, 1.0


def device_activations(N: int, K: int, seed: int, stream: int, device="cuda"):
    import torch
    gen = _torch_gen(seed, stream, device)
    return torch.randn((N, K), generator=gen, device=device).half()


# ---------------------------------------------------------------------------
# Workload shapes (Qwen3-4B-shaped decode layer and the sweeps around it).
# ---------------------------------------------------------------------------

#: single small GEMV
CONFIG0 = dict(name="q4k_gemv_256x2560", qtype=Q4_K, M=256, K=2560, N=1)

#: one decode layer: (role, type, M, K)
LAYER = [
    ("wq", Q4_K, 4096, 2560),
    ("wk", Q4_K, 1024, 2560),
    ("wv", Q6_K, 1024, 2560),
    ("wo", Q4_K, 2560, 4096),
    ("gate", Q4_K, 9728, 2560),
    ("up", Q4_K, 9728, 2560),
    ("down", Q6_K, 2560, 9728),
]

#: skinny row sweep
SWEEP_SHAPES = [(Q4_K, 9728, 2560), (Q5_K, 2560, 9728)]
SWEEP_N = [1, 2, 4, 8, 16, 32]

#: prefill chunk sizes over the 36-layer set
PREFILL_N = [33, 64, 128]
N_LAYERS = 36

#: NVFP4 shapes and row counts
NVFP4_SHAPES = [(27648, 5120), (5120, 27648), (7168, 5120)]
NVFP4_N = [1, 8, 16, 32]
