"""fp64 CPU oracle of the routed-expert MXFP4 MoE layer -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
import this package.  It shares no code with the CUDA path: the arithmetic is
in `moe_oracle.c` (plain C, fp64), driven from here with numpy for marshalling,
and the only common module is `synth` (seeded inputs, no method arithmetic).

Readings of the pages this oracle encodes (Deltafin pages: "工作原理" -- the
router picks 16 experts per layer per token; "Deltafin 的功能" -- experts used at
their released MXFP4 precision, one 17.5 MiB record per (layer, expert);
"作者仍需帮助的事项" -- expert-major prefill reading each expert once for all
routed rows):

  * route: exact logits, top-k with ties to the lower index, descending order,
    softmax over the k selected logits (fp64);
  * expert: g = W_g x, u = W_u x, h = silu(g) * u, o = W_d h (fp64), MXFP4 weights
    dequantised as E2M1(code) * 2^(scale - 127);
  * combine: y = sum_j w_j o_j (+ residual), fp64, unrounded;
  * prefill: the token->expert permutation is the stable sort of the pairs
    p = t*k + j by expert; with MXFP8 activations x and h are quantised per
    32-block (OCP MX rule) before the contractions that consume them;
  * stacked layers: x_hat = x * 2^-p (p = floor(log2 amax|x|) - 2, exact),
    x_next = bf16(x + MoE(x_hat)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from collections import OrderedDict

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no GPU involved)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
             "-o", _SO, _SRC, "-lm"])
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        L.orc_splitmix64_at.restype = ctypes.c_uint64
        L.orc_splitmix64_at.argtypes = [ctypes.c_uint64] * 2
        L.orc_u64.restype = ctypes.c_uint64
        L.orc_u64.argtypes = [ctypes.c_uint64] * 3
        L.orc_gen_expert.restype = None
        L.orc_gen_expert.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u8p, _u8p]
        L.orc_e2m1_value.restype = ctypes.c_double
        L.orc_e2m1_value.argtypes = [ctypes.c_uint]
        L.orc_e8m0_value.restype = ctypes.c_double
        L.orc_e8m0_value.argtypes = [ctypes.c_uint]
        L.orc_e4m3_value.restype = ctypes.c_double
        L.orc_e4m3_value.argtypes = [ctypes.c_uint]
        L.orc_e4m3_encode.restype = ctypes.c_uint
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_quant_mxfp8.restype = None
        L.orc_quant_mxfp8.argtypes = [_f64p, ctypes.c_int, _u8p, _u8p, _f64p]
        L.orc_bf16_value.restype = ctypes.c_double
        L.orc_bf16_value.argtypes = [ctypes.c_uint16]
        L.orc_bf16_round.restype = ctypes.c_uint16
        L.orc_bf16_round.argtypes = [ctypes.c_double]
        L.orc_route.restype = ctypes.c_int
        L.orc_route.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, _u16p, ctypes.c_int,
                                ctypes.c_void_p, ctypes.c_int, _i32p, _f64p, ctypes.c_void_p]
        L.orc_expert_forward.restype = None
        L.orc_expert_forward.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_int, _f64p, ctypes.c_int,
                                         _f64p, ctypes.c_void_p, ctypes.c_int]
        L.orc_mxfp8_ambiguity.restype = None
        L.orc_mxfp8_ambiguity.argtypes = [_f64p, _f64p, ctypes.c_int, _f64p]
        L.orc_expert_ambiguity.restype = None
        L.orc_expert_ambiguity.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_int, _f64p, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_int, _f64p]
        L.orc_mx_ambiguity.restype = None
        L.orc_mx_ambiguity.argtypes = [_f64p, _f64p, ctypes.c_int, ctypes.c_int, _f64p]
        L.orc_e2m1_encode.restype = ctypes.c_uint
        L.orc_e2m1_encode.argtypes = [ctypes.c_double]
        L.orc_quant_mxfp4.restype = None
        L.orc_quant_mxfp4.argtypes = [_f64p, ctypes.c_int, _u8p, _u8p, _f64p]
        L.orc_h_radius.restype = None
        L.orc_h_radius.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_int, _f64p, ctypes.c_int, ctypes.c_double,
                                   _f64p, _f64p]
        L.orc_set_threads.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_prescale_exponent.restype = ctypes.c_int
        L.orc_prescale_exponent.argtypes = [_u16p, ctypes.c_int]
        L.orc_prescale.restype = None
        L.orc_prescale.argtypes = [_u16p, ctypes.c_int, _u16p]
        _lib = L
    return _lib


# ------------------------------------------------------------------ primitives


def set_threads(n: int) -> int:
    """Threads of the oracle's OpenMP loops (n <= 0 leaves it); returns the previous count."""
    return int(lib().orc_set_threads(n))


def splitmix64_at(state: int, i: int) -> int:
    return int(lib().orc_splitmix64_at(state, i))


def u64(seed: int, stream: int, i: int) -> int:
    return int(lib().orc_u64(seed, stream, i))


def gen_expert(seed: int, e: int, H: int, I: int):
    """Logical MXFP4 bytes of expert e: (codes [3*H*I/2], scales [3*H*I/32])."""
    codes = np.empty(3 * H * I // 2, dtype=np.uint8)
    scales = np.empty(3 * H * I // 32, dtype=np.uint8)
    lib().orc_gen_expert(seed, e, H, I, codes, scales)
    return codes, scales


def e2m1_value(code: int) -> float:
    return float(lib().orc_e2m1_value(code))


def e8m0_value(b: int) -> float:
    return float(lib().orc_e8m0_value(b))


def e4m3_value(c: int) -> float:
    return float(lib().orc_e4m3_value(c))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def quant_mxfp8(v: np.ndarray):
    """MXFP8 (E4M3 + E8M0 per 32) of a 1-D vector: (codes, scale bytes, dequantised)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    n = v.size
    codes = np.empty(n, dtype=np.uint8)
    sb = np.empty((n + 31) // 32, dtype=np.uint8)
    deq = np.empty(n, dtype=np.float64)
    lib().orc_quant_mxfp8(v, n, codes, sb, deq)
    return codes, sb, deq


def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(v)))


def quant_mxfp4(v: np.ndarray):
    """MXFP4 (E2M1 + E8M0 per 32) of a 1-D vector: (codes, scale bytes, dequantised)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    n = v.size
    codes = np.empty(n, dtype=np.uint8)
    sb = np.empty((n + 31) // 32, dtype=np.uint8)
    deq = np.empty(n, dtype=np.float64)
    lib().orc_quant_mxfp4(v, n, codes, sb, deq)
    return codes, sb, deq


def bf16_value(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_round(v) -> np.ndarray:
    """Round doubles to bf16 bits, nearest-even, without intermediate fp32."""
    L = lib()
    a = np.asarray(v, dtype=np.float64)
    out = np.fromiter((L.orc_bf16_round(float(t)) for t in a.ravel()), dtype=np.uint16, count=a.size)
    return out.reshape(a.shape)


def route(x_bits: np.ndarray, Wr_bits: np.ndarray, k: int, skew: np.ndarray | None = None):
    """Exact routing of M tokens: (idx int32 [M,k], w fp64 [M,k], logits fp64 [M,E])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    W = np.ascontiguousarray(Wr_bits, dtype=np.uint16)
    M, H = x.shape
    E = W.shape[0]
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float64)
    logits = np.empty((M, E), dtype=np.float64)
    sk = None
    if skew is not None:
        sk = np.ascontiguousarray(skew, dtype=np.float32)
    rc = lib().orc_route(x, M, H, W, E, sk.ctypes.data if sk is not None else None, k, idx, w,
                         logits.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle route failed ({rc})")
    return idx, w, logits


def expert_forward(codes: np.ndarray, scales: np.ndarray, H: int, I: int, x: np.ndarray,
                   h_mode: int = 0):
    """One expert applied to rows x [n,H] (fp64): (o [n,H], h [n,I])."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    n = x.shape[0]
    y = np.empty((n, H), dtype=np.float64)
    h = np.empty((n, I), dtype=np.float64)
    lib().orc_expert_forward(np.ascontiguousarray(codes, dtype=np.uint8),
                             np.ascontiguousarray(scales, dtype=np.uint8), H, I, x, n, y,
                             h.ctypes.data, h_mode)
    return y, h


# Error model of the fp32 h of the tensor-core path (orc_h_radius): each
# block-scaled MMA step of K = 32 adds its exact block sum S_t to the fp32
# accumulator P_{t-1} with an error of at most this times |P_{t-1}| + |S_t| (one
# fp32 ulp of the larger operand), so |g_gpu - g| <= MMA_STEP_REL *
# sum_t (|P_{t-1}| + |S_t|).
MMA_STEP_REL = 2.0 ** -23


def mxfp8_ambiguity(v: np.ndarray, radius) -> np.ndarray:
    """delta[i]: change an alternative MXFP8 rounding may make when v[i] is known
    only to within radius[i] (absolute)."""
    return mx_ambiguity(v, radius, 8)


def mx_ambiguity(v: np.ndarray, radius, fmt: int) -> np.ndarray:
    """As mxfp8_ambiguity for fmt 8 (MXFP8) or 4 (MXFP4)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    r = np.ascontiguousarray(np.broadcast_to(radius, v.shape), dtype=np.float64)
    d = np.empty_like(v)
    lib().orc_mx_ambiguity(v, r, v.size, fmt, d)
    return d


def h_radius(codes: np.ndarray, scales: np.ndarray, H: int, I: int, x: np.ndarray,
             rel: float = MMA_STEP_REL):
    """h [n, I] of one expert for MXFP8-exact rows x [n, H], and the error radius of
    the fp32 h the tensor-core path computes under the step-error model `rel`."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    n = x.shape[0]
    h = np.empty((n, I), dtype=np.float64)
    r = np.empty((n, I), dtype=np.float64)
    lib().orc_h_radius(np.ascontiguousarray(codes, dtype=np.uint8), np.ascontiguousarray(scales, dtype=np.uint8),
                       H, I, x, n, rel, h, r)
    return h, r


def prescale(x_bits: np.ndarray) -> np.ndarray:
    """Row-wise exact power-of-two pre-scale (bf16 bits in, bf16 bits out)."""
    x = np.ascontiguousarray(np.atleast_2d(x_bits), dtype=np.uint16)
    out = np.empty_like(x)
    for r in range(x.shape[0]):
        row = np.ascontiguousarray(x[r])
        o = np.empty_like(row)
        lib().orc_prescale(row, row.size, o)
        out[r] = o
    return out.reshape(np.shape(x_bits))


# ---------------------------------------------------------------- the layer


class SyntheticPool:
    """Experts of one seeded pool, generated on demand by the oracle's own SplitMix64."""

    def __init__(self, seed: int, E: int, H: int, I: int, cache: int = 32):
        self.seed, self.E, self.H, self.I = seed, E, H, I
        self._cache: OrderedDict = OrderedDict()
        self._cap = cache

    def __call__(self, e: int):
        if e in self._cache:
            self._cache.move_to_end(e)
            return self._cache[e]
        v = gen_expert(self.seed, e, self.H, self.I)
        self._cache[e] = v
        if len(self._cache) > self._cap:
            self._cache.popitem(last=False)
        return v


def pair_outputs(experts, H: int, I: int, x: np.ndarray, idx: np.ndarray, h_mode: int = 0) -> np.ndarray:
    """Unweighted expert outputs o[m, j] = expert_{idx[m,j]}(x[m]) (fp64 [M, k, H])."""
    M, k = idx.shape
    o = np.zeros((M, k, H), dtype=np.float64)
    for e in sorted(set(int(v) for v in idx.ravel())):
        rows = [(m, j) for m in range(M) for j in range(k) if idx[m, j] == e]
        codes, scales = experts(e)
        ye, _ = expert_forward(codes, scales, H, I, np.stack([x[m] for m, _ in rows]), h_mode)
        for r, (m, j) in enumerate(rows):
            o[m, j] = ye[r]
    return o


def combine_rows(experts, H: int, I: int, x: np.ndarray, idx: np.ndarray, w: np.ndarray,
                 h_mode: int = 0) -> np.ndarray:
    """y[m] = sum_j w[m,j] * expert_{idx[m,j]}(x[m]) in fp64, each distinct expert
    applied once to all rows routed to it, the sum taken in slot order j."""
    M, k = idx.shape
    o = np.zeros((M, k, H), dtype=np.float64)
    for e in sorted(set(int(v) for v in idx.ravel())):
        rows = [(m, j) for m in range(M) for j in range(k) if idx[m, j] == e]
        codes, scales = experts(e)
        xe = np.stack([x[m] for m, _ in rows])
        ye, _ = expert_forward(codes, scales, H, I, xe, h_mode)
        for r, (m, j) in enumerate(rows):
            o[m, j] = ye[r]
    y = np.zeros((M, H), dtype=np.float64)
    for j in range(k):
        y += w[:, j:j + 1] * o[:, j]
    return y


def decode_layer(experts, x_bits: np.ndarray, Wr_bits: np.ndarray, k: int,
                 skew: np.ndarray | None = None, residual_bits: np.ndarray | None = None):
    """Decode/verify forward of M rows: dict(idx, w, y fp64 [M,H], union)."""
    x_bits = np.atleast_2d(x_bits)
    H = x_bits.shape[1]
    I = experts.I
    idx, w, logits = route(x_bits, Wr_bits, k, skew)
    y = combine_rows(experts, H, I, bf16_value(x_bits), idx, w)
    if residual_bits is not None:
        y = y + bf16_value(residual_bits)
    return {"idx": idx, "w": w, "y": y, "logits": logits,
            "union": sorted(set(int(v) for v in idx.ravel()))}


def sort_pairs(idx: np.ndarray, E: int):
    """Expert-major order of the (token, slot) pairs p = t*k + j.

    perm[r] = the pair at sorted position r, sorted by (expert, p) -- a stable sort
    of p by expert; inv_perm[p] = its position; offsets[e] = first position of e."""
    T, k = idx.shape
    keys = idx.reshape(-1).astype(np.int64)
    perm = np.argsort(keys, kind="stable").astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    counts = np.bincount(keys, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return perm, inv, offsets


def pair_ambiguity(experts, H: int, I: int, x: np.ndarray, idx: np.ndarray,
                   eps: float = MMA_STEP_REL, fmt: int = 8) -> np.ndarray:
    """amb[m, j, o]: the largest change of expert_{idx[m,j]}(x[m])[o] that an
    alternative (equally correct) MX rounding of its h could make (fmt 8: MXFP8,
    4: MXFP4)."""
    M, k = idx.shape
    amb = np.zeros((M, k, H), dtype=np.float64)
    for e in sorted(set(int(v) for v in idx.ravel())):
        rows = [(m, j) for m in range(M) for j in range(k) if idx[m, j] == e]
        codes, scales = experts(e)
        xe = np.ascontiguousarray(np.stack([x[m] for m, _ in rows]), dtype=np.float64)
        ya = np.empty((len(rows), H), dtype=np.float64)
        lib().orc_expert_ambiguity(np.ascontiguousarray(codes), np.ascontiguousarray(scales), H, I, xe, len(rows),
                                   eps, fmt, ya)
        for r, (m, j) in enumerate(rows):
            amb[m, j] = ya[r]
    return amb


def combine_ambiguity(experts, H: int, I: int, x: np.ndarray, idx: np.ndarray, w: np.ndarray,
                      eps: float = MMA_STEP_REL, fmt: int = 8) -> np.ndarray:
    """Per output, sum_j |w_j| * pair_ambiguity: the part of the difference between
    two correct MX-h layer outputs that rounding choices can explain."""
    amb = pair_ambiguity(experts, H, I, x, idx, eps, fmt)
    return np.einsum("mj,mjh->mh", np.abs(w), amb)


def quant_rows_mxfp8(x: np.ndarray) -> np.ndarray:
    """Rows of x (fp64) replaced by their MXFP8-dequantised values."""
    out = np.empty_like(x, dtype=np.float64)
    for r in range(x.shape[0]):
        out[r] = quant_mxfp8(x[r])[2]
    return out


def quant_rows_mxfp4(x: np.ndarray) -> np.ndarray:
    """Rows of x (fp64) replaced by their MXFP4-dequantised values."""
    out = np.empty_like(x, dtype=np.float64)
    for r in range(x.shape[0]):
        out[r] = quant_mxfp4(x[r])[2]
    return out


def quant_rows(x: np.ndarray, act_mode: int) -> np.ndarray:
    """The activation rows as the prefill path quantises them: act_mode 1 MXFP8,
    2 MXFP4, 0 unquantised."""
    if act_mode == 1:
        return quant_rows_mxfp8(x)
    if act_mode == 2:
        return quant_rows_mxfp4(x)
    return np.asarray(x, dtype=np.float64)


def prefill_layer(experts, x_bits: np.ndarray, Wr_bits: np.ndarray, k: int, act_mode: int = 1,
                  sample_tokens=None):
    """Expert-major prefill: routing and the pair permutation for all T tokens, and
    the output y for the tokens in `sample_tokens` (all when None).

    act_mode 1: activations MXFP8 (x before W_g/W_u, h before W_d); 2: MXFP4 (the
    same two steps with E2M1 elements); 0: fp64."""
    T, H = x_bits.shape
    idx, w, _ = route(x_bits, Wr_bits, k)
    perm, inv, offsets = sort_pairs(idx, experts.E)
    toks = np.arange(T) if sample_tokens is None else np.asarray(sample_tokens)
    xs = quant_rows(bf16_value(x_bits[toks]), act_mode)
    y = combine_rows(experts, H, experts.I, xs, idx[toks], w[toks], h_mode=act_mode)
    amb = (combine_ambiguity(experts, H, experts.I, xs, idx[toks], w[toks], fmt=8 if act_mode == 1 else 4)
           if act_mode in (1, 2) else np.zeros_like(y))
    return {"idx": idx, "w": w, "perm": perm, "inv_perm": inv, "offsets": offsets,
            "tokens": toks, "y": y, "y_amb": amb}


def stacked_step(pools, routers, skews, x_bits: np.ndarray, k: int):
    """One token through L stacked layers (pre-scale, route, experts, residual add).

    Returns per-layer dicts with the layer input x_l (bf16 bits), x_hat_l, idx, w
    and y_l, and the final bf16 output."""
    x = np.atleast_2d(x_bits).astype(np.uint16)
    layers = []
    for pool, Wr, sk in zip(pools, routers, skews):
        xh = prescale(x)
        d = decode_layer(pool, xh, Wr, k, sk)
        x_next = bf16_round(bf16_value(x) + d["y"])
        layers.append({"x": x, "x_hat": xh, "idx": d["idx"], "w": d["w"], "y": d["y"],
                       "x_next": x_next})
        x = x_next
    return layers, x
