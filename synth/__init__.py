"""Seeded synthetic inputs for the routed-expert MXFP4 MoE layer.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.  It
holds no arithmetic of the method itself (no routing, no dequantisation, no
matmul): only the counter-based random generator, the workload shapes and the
recipes that turn random bits into bf16 activations, router weights and the
per-expert popularity skew.

Counter-based generator
-----------------------
SplitMix64 (Steele, Lea & Flood, "Fast Splittable Pseudorandom Number
Generators", OOPSLA 2014), used in counter mode:

    mix64(z)      = the SplitMix64 output finaliser
    key(seed, s)  = mix64(mix64(seed + G) ^ mix64(s + 2G))
    u64(seed,s,i) = mix64(key(seed, s) + (i + 1) * G)       (all mod 2^64)

so u64(seed, s, 0..) is the SplitMix64 output sequence whose state starts at
key(seed, s).  The resident expert pool is drawn from the same definition by a
device kernel (pool codes: stream 2e, scale bytes: stream 2e+1); the CPU oracle
has its own C implementation of it.

Workloads (the five configurations of the routed-expert layer)
--------------------------------------------------------------
  tiny      E=64,  H=1024, I=512,  k=16, decode of 1 token
  full      E=896, H=7168, I=1600, k=16, decode of 1 token (1000 tokens)
  stacked   8 full-size layers, Zipf(1.1) popularity skew, residual, 256 tokens
  verify    full-size layer, M in {2,5,9,17} correlated rows, 100 batches each
  prefill   full-size layer, T in {512, 2048, 8192} tokens, MXFP8 activations
"""
from __future__ import annotations

import dataclasses

import numpy as np

G = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1

# ---------------------------------------------------------------- SplitMix64


def mix64_int(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def key_int(seed: int, stream: int) -> int:
    return mix64_int(mix64_int(seed + G) ^ mix64_int(stream + 2 * G))


def u64_int(seed: int, stream: int, i: int) -> int:
    return mix64_int(key_int(seed, stream) + (i + 1) * G)


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(0xBF58476D1CE4E5B9)
        z ^= z >> np.uint64(27)
        z *= np.uint64(0x94D049BB133111EB)
        z ^= z >> np.uint64(31)
    return z


def u64_array(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """u64(seed, stream, start .. start+count-1) as a uint64 array."""
    key = np.uint64(key_int(seed, stream))
    i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + i * np.uint64(G)
    return _mix64_np(z)


# ------------------------------------------------------------ bf16 helpers


def bf16_bits_from_f64(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of `v`: round to fp32 (RNE), then fp32 -> bf16 (RNE).

    This two-step rounding is part of the input recipe only; the method's own
    roundings are defined elsewhere.
    """
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ------------------------------------------------------------- samplers


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in (0, 1): ((u >> 11) + 0.5) * 2^-53."""
    u = u64_array(seed, stream, start, count)
    return ((u >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal_f64(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals by Box-Muller on uniform pairs (2i, 2i+1) of one stream."""
    npair = (n + 1) // 2
    u = uniform01(seed, stream, 0, 2 * npair)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    t = 2.0 * np.pi * u[1::2]
    z = np.empty(2 * npair, dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    return z[:n]


# ------------------------------------------------------------- workloads


@dataclasses.dataclass(frozen=True)
class Shape:
    E: int
    H: int
    I: int
    k: int = 16


TINY = Shape(E=64, H=1024, I=512, k=16)
FULL = Shape(E=896, H=7168, I=1600, k=16)

VERIFY_M = (2, 5, 9, 17)
PREFILL_T = (512, 2048, 8192)
PREFILL_T_LARGE = (16384, 32768)    # the large-T sweep of the MXFP4-activation prefill
STACKED_LAYERS = 8
ZIPF_S = 1.1
VERIFY_MIX = 0.7


def pool_seed(layer: int) -> int:
    return 1000 * layer + 1


def router_seed(layer: int) -> int:
    return 1000 * layer + 2


def skew_seed(layer: int) -> int:
    return 1000 * layer + 3


# seeds of the token streams, one per workload
TOKENS_SEED = {"tiny": 0, "full": 0, "stacked": 10, "verify": 20, "prefill": 30}


def expert_code_bytes(H: int, I: int) -> int:
    """Packed E2M1 bytes of one expert: gate [I,H] + up [I,H] + down [H,I], 2 per byte."""
    return 3 * H * I // 2


def expert_scale_bytes(H: int, I: int) -> int:
    """E8M0 bytes of one expert: one per 32 elements along K."""
    return 3 * H * I // 32


def tokens_bf16(seed: int, t0: int, T: int, H: int) -> np.ndarray:
    """Tokens t0..t0+T-1, each ~N(0,1) from stream t, as bf16 bits [T, H]."""
    out = np.empty((T, H), dtype=np.uint16)
    for t in range(T):
        out[t] = bf16_bits_from_f64(normal_f64(seed, t0 + t, H))
    return out


def router_bf16(seed: int, E: int, H: int) -> np.ndarray:
    """Router weights W_r[e, h] ~ N(0, 1/H) as bf16 bits [E, H]; row e from stream e."""
    out = np.empty((E, H), dtype=np.uint16)
    s = 1.0 / np.sqrt(H)
    for e in range(E):
        out[e] = bf16_bits_from_f64(normal_f64(seed, e, H) * s)
    return out


def zipf_skew_f32(seed: int, E: int, s: float = ZIPF_S) -> np.ndarray:
    """Per-expert additive logit skew from a Zipf(s) popularity law.

    A seeded permutation gives each expert a rank r in 1..E (sort of u64(seed, 0, e),
    ties impossible in practice and broken by index); skew_e = fp32(-s * ln r_e), so
    exp(skew) is proportional to r^-s.
    """
    keys = u64_array(seed, 0, 0, E)
    order = np.argsort(keys, kind="stable")
    rank = np.empty(E, dtype=np.int64)
    rank[order] = np.arange(1, E + 1)
    return (-s * np.log(rank.astype(np.float64))).astype(np.float32)


def verify_batch_bf16(seed: int, batch: int, M: int, H: int, mix: float = VERIFY_MIX) -> np.ndarray:
    """M correlated rows: x_m = mix * s + sqrt(1 - mix^2) * z_m, each N(0,1), bf16 bits [M, H].

    Shared vector s from stream 64*batch + 63, row m's own z_m from stream 64*batch + m.
    """
    shared = normal_f64(seed, 64 * batch + 63, H)
    c = np.sqrt(1.0 - mix * mix)
    out = np.empty((M, H), dtype=np.uint16)
    for m in range(M):
        out[m] = bf16_bits_from_f64(mix * shared + c * normal_f64(seed, 64 * batch + m, H))
    return out
