"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test fixes one piece of the oracle against something independent: a
published value (golden files with citations), a closed form, a library routine,
an invariant, or brute force over exact rationals on tiny inputs.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from tests._util import dequant_mxfp4 as _dequant, split_expert as _split

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split("#")[0].strip() for ln in f if ln.split("#")[0].strip()]


# ------------------------------------------------------------------ generator


def test_splitmix64_published_vectors():
    for ln in _golden_lines("splitmix64_vectors.txt"):
        state, i, out = ln.split()
        assert oracle.splitmix64_at(int(state), int(i)) == int(out, 16)
        assert synth.mix64_int(int(state) + (int(i) + 1) * synth.G) == int(out, 16)


def test_counter_mode_two_implementations_agree():
    for seed, stream, i in [(0, 0, 0), (1, 7, 12345), (2**63 + 5, 2**40, 2**33), (1001, 1791, 99)]:
        assert oracle.u64(seed, stream, i) == synth.u64_int(seed, stream, i)
    arr = synth.u64_array(3, 9, 100, 50)
    assert [int(v) for v in arr] == [oracle.u64(3, 9, 100 + j) for j in range(50)]


def test_generated_expert_bytes_follow_the_recipe():
    H, I = 64, 32
    codes, scales = oracle.gen_expert(1, 5, H, I)
    assert codes.size == 3 * H * I // 2 and scales.size == 3 * H * I // 32
    for b in [0, 1, 7, 8, 100, codes.size - 1]:
        r = synth.u64_int(1, 10, b // 8)
        assert codes[b] == (r >> (8 * (b % 8))) & 0xFF
    for j in [0, 3, scales.size - 1]:
        assert scales[j] == 118 + (synth.u64_int(1, 11, j) >> 32) % 5
    big_c, big_s = oracle.gen_expert(7, 3, 1024, 512)
    assert set(np.unique(big_s)) == {118, 119, 120, 121, 122}
    nib = np.concatenate([big_c & 15, big_c >> 4])
    hist = np.bincount(nib, minlength=16) / nib.size
    assert np.all(np.abs(hist - 1 / 16) < 0.002)


# ----------------------------------------------------------------- MX formats


def test_e2m1_table_from_spec_and_bitfields():
    rows = [ln.split() for ln in _golden_lines("e2m1_e8m0.txt")]
    for r in rows:
        if r[0] == "e8m0":
            b, v = int(r[1]), float(r[2])
            assert oracle.e8m0_value(b) == v
            continue
        code, v = int(r[0]), float(r[1])
        got = oracle.e2m1_value(code)
        assert got == v and math.copysign(1, got) == math.copysign(1, v)
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        bits = (m * 0.5) if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert got == (-bits if s else bits)


def test_e8m0_all_bytes():
    for b in range(255):
        assert oracle.e8m0_value(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_e4m3_values_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(tv[c]):
            assert math.isnan(v)
        else:
            assert v == tv[c]


def test_e4m3_encode_round_trip_midpoints_and_saturation():
    finite = [c for c in range(127)]
    vals = [oracle.e4m3_value(c) for c in finite]
    for c, v in zip(finite, vals):
        assert oracle.e4m3_encode(v) == c
        assert oracle.e4m3_encode(-v) == (c | 0x80)
    for c in range(126):                        # exact midpoints go to the even code
        mid = (vals[c] + vals[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want
        # just off the midpoint goes to the nearer neighbour
        eps = (vals[c + 1] - vals[c]) * 1e-6
        assert oracle.e4m3_encode(mid - eps) == c
        assert oracle.e4m3_encode(mid + eps) == c + 1
    for big in [448.0, 449.0, 464.0, 480.0, 1e6, 1e300]:
        assert oracle.e4m3_encode(big) == 0x7E
        assert oracle.e4m3_encode(-big) == 0xFE


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(4000) * np.exp2(rng.integers(-12, 8, size=4000))
    v = v[np.abs(v) < 440].astype(np.float32).astype(np.float64)   # fp32-exact, in range
    t = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for a, c in zip(v, t):
        assert oracle.e4m3_encode(a) == c


def test_e4m3_encode_every_bf16_pattern_by_brute_force():
    """E4M3 encoding (round to nearest, ties to the even code, saturating at 448) of
    every finite bf16 value, against a nearest-value search over the 127 magnitudes
    written out from the format's definition (bias 7, 3 mantissa bits, subnormals at
    exponent field 0, magnitude code 0x7F reserved for NaN)."""
    mags = np.array([(m & 7) / 8.0 * 2.0 ** -6 if (m >> 3) == 0 else (1 + (m & 7) / 8.0) * 2.0 ** ((m >> 3) - 7)
                     for m in range(127)])
    assert mags[-1] == 448.0 and np.all(np.diff(mags) > 0)
    bits = np.arange(65536, dtype=np.uint32)
    f32 = (bits << 16).view(np.float32)
    finite = np.isfinite(f32)
    vals = np.where(finite, f32, 0).astype(np.float64)
    for b, v in zip(bits[finite], vals[finite]):
        a = abs(v)
        if a >= 448.0:
            m = 126
        else:
            hi = int(np.searchsorted(mags, a))          # first magnitude >= a
            lo = max(hi - 1, 0)
            dl, dh = a - mags[lo], mags[hi] - a
            m = lo if dl < dh else hi if dh < dl else (lo if lo % 2 == 0 else hi)
        want = m | (0x80 if (b >> 15) & 1 else 0)
        assert oracle.e4m3_encode(v) == want, (hex(int(b)), v)


def test_mxfp8_block_rule():
    # amax 1.0 -> X = floor(log2 1) - 8 = -8 (byte 119); 1.0 -> 256 -> code exact
    v = np.zeros(64)
    v[0] = 1.0
    v[5] = -0.75
    v[32] = 500.0         # X = 8 - 8 = 0; 500 saturates to 448
    v[33] = 3.0
    codes, sb, deq = oracle.quant_mxfp8(v)
    assert list(sb) == [119, 127]
    assert deq[0] == 1.0 and deq[5] == -0.75
    assert deq[32] == 448.0 and deq[33] == 3.0
    z = oracle.quant_mxfp8(np.zeros(32))
    assert z[1][0] == 0 and np.all(z[2] == 0)


def test_mxfp8_error_bound_on_bf16_inputs():
    # every element of a block is within half an E4M3 step of its value, the step
    # being 2^(X + e - 3) for element exponent e >= -6 (relative 2^-4 at most)
    x = synth.bf16_bits_to_f64(synth.tokens_bf16(0, 0, 4, 1024)).ravel()
    _, sb, deq = oracle.quant_mxfp8(x)
    for b in range(0, x.size, 32):
        X = int(sb[b // 32]) - 127
        amax = np.max(np.abs(x[b:b + 32]))
        assert 256 <= amax / 2.0 ** X < 512
        err = np.abs(deq[b:b + 32] - x[b:b + 32])
        bound = np.maximum(np.abs(x[b:b + 32]) * 2.0 ** -4, 2.0 ** (X - 10))
        small = np.abs(x[b:b + 32]) / 2.0 ** X <= 448
        assert np.all(err[small] <= bound[small])


def test_bf16_round_against_fp32_path():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(3000) * np.exp2(rng.integers(-140, 120, size=3000))).astype(np.float32)
    v = v.astype(np.float64)                    # fp32-exact values: one rounding either way
    got = oracle.bf16_round(v)
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert oracle.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80       # tie -> even
    assert oracle.bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82   # tie -> even (up)
    assert oracle.bf16_round(np.array([1e39]))[0] == 0x7F80


# -------------------------------------------------------------------- routing


def _bf16(rng, shape, scale=1.0):
    return synth.bf16_bits_from_f64(rng.standard_normal(shape) * scale)


def _brute_route(x_bits, W_bits, k, skew=None):
    """Exact logits as rationals, sort by (-value, index)."""
    x = [Fraction(float(v)) for v in synth.bf16_bits_to_f64(x_bits)]
    out = []
    for e in range(W_bits.shape[0]):
        w = [Fraction(float(v)) for v in synth.bf16_bits_to_f64(W_bits[e])]
        s = sum(a * b for a, b in zip(x, w))
        if skew is not None:
            s += Fraction(float(skew[e]))
        out.append(s)
    order = sorted(range(len(out)), key=lambda e: (-out[e], e))
    return order[:k], out


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_route_matches_exact_rationals(seed):
    rng = np.random.default_rng(seed)
    E, H = 24, 48
    x = _bf16(rng, (3, H))
    W = _bf16(rng, (E, H), 1 / np.sqrt(H))
    skew = (rng.standard_normal(E) * 0.1).astype(np.float32) if seed % 2 else None
    for k in (1, 5, 16, E):
        idx, w, logits = oracle.route(x, W, k, skew)
        for m in range(3):
            want, exact = _brute_route(x[m], W, k, skew)
            assert list(idx[m]) == want
            # logits are the exact values rounded once to double
            assert all(logits[m, e] == float(exact[e]) for e in range(E))
            z = [math.exp(float(exact[e]) - float(exact[want[0]])) for e in want]
            assert np.allclose(w[m], np.array(z) / sum(z), rtol=1e-14, atol=0)


def test_route_planted_ties_and_near_ties():
    rng = np.random.default_rng(7)
    E, H = 20, 64
    x = _bf16(rng, (1, H))
    W = _bf16(rng, (E, H), 1 / np.sqrt(H))
    # make experts 3, 11, 17 the clear winners and exactly equal: 11 is 3 with its
    # elements permuted in pairs of equal x (same multiset of products) -> exact tie
    W[3] = synth.bf16_bits_from_f64(np.sign(synth.bf16_bits_to_f64(x[0])) * 0.5)
    W[11] = W[3]
    W[17] = W[3]
    # expert 5: expert 3 with one element nudged by one bf16 ulp -> near tie
    W[5] = W[3]
    W[5, 10] = W[5, 10] + 1 if synth.bf16_bits_to_f64(x[0, 10]) > 0 else W[5, 10] - 1
    idx, w, logits = oracle.route(x, W, 6)
    want, exact = _brute_route(x[0], W, 6)
    assert list(idx[0]) == want
    assert exact[3] == exact[11] == exact[17] and exact[5] != exact[3]
    pos = list(idx[0])
    assert pos.index(3) < pos.index(11) < pos.index(17)     # ties -> lower index first
    assert w[0, pos.index(3)] == w[0, pos.index(11)]


def test_route_weights_sum_to_one_and_are_monotone():
    x = synth.tokens_bf16(0, 0, 5, 1024)
    W = synth.router_bf16(2, 64, 1024)
    idx, w, logits = oracle.route(x, W, 16)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-15)
    for m in range(5):
        l = logits[m, idx[m]]
        assert np.all(np.diff(l) <= 0) and np.all(np.diff(w[m]) <= 0)


# ------------------------------------------------------------------ the expert


def test_zero_code_expert_contributes_zero():
    H, I = 256, 128
    codes = np.zeros(3 * H * I // 2, dtype=np.uint8)
    scales = np.full(3 * H * I // 32, 120, dtype=np.uint8)
    x = synth.bf16_bits_to_f64(synth.tokens_bf16(0, 0, 2, H))
    y, h = oracle.expert_forward(codes, scales, H, I, x)
    assert np.all(y == 0.0) and np.all(h == 0.0)
    codes8 = np.full_like(codes, 0x88)          # -0 codes
    y, h = oracle.expert_forward(codes8, scales, H, I, x)
    assert np.all(y == 0.0)


def test_all_ones_closed_form():
    # every code 2 (value 1.0), every scale byte 127 (2^0): each gate and up row is
    # s = sum(x), h = silu(s) * s for every i, and every output is I * h
    H, I = 512, 256
    codes = np.full(3 * H * I // 2, 0x22, dtype=np.uint8)
    scales = np.full(3 * H * I // 32, 127, dtype=np.uint8)
    x = synth.bf16_bits_to_f64(synth.tokens_bf16(0, 3, 1, H)) / 8
    s = math.fsum(x[0])
    hval = s / (1 + math.exp(-s)) * s
    y, h = oracle.expert_forward(codes, scales, H, I, x)
    assert np.allclose(h, hval, rtol=1e-13, atol=0)
    assert np.allclose(y, I * hval, rtol=1e-13, atol=0)


def test_expert_matches_dense_dequantised_matmul():
    H, I = 128, 64
    codes, scales = oracle.gen_expert(11, 2, H, I)
    (cg, sg), (cu, su), (cd, sd) = _split(codes, scales, H, I)
    Wg, Wu, Wd = _dequant(cg, sg, I, H), _dequant(cu, su, I, H), _dequant(cd, sd, H, I)
    x = synth.bf16_bits_to_f64(synth.tokens_bf16(4, 0, 3, H))
    g, u = x @ Wg.T, x @ Wu.T
    h_ref = g / (1 + np.exp(-g)) * u
    y_ref = h_ref @ Wd.T
    y, h = oracle.expert_forward(codes, scales, H, I, x)
    assert np.allclose(h, h_ref, rtol=1e-12, atol=1e-12 * np.abs(h_ref).max())
    assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-12 * np.abs(y_ref).max())


def test_power_of_two_linearity_of_down_scales():
    H, I = 128, 64
    codes, scales = oracle.gen_expert(5, 1, H, I)
    x = synth.bf16_bits_to_f64(synth.tokens_bf16(0, 0, 1, H))
    y1, h1 = oracle.expert_forward(codes, scales, H, I, x)
    s2 = scales.copy()
    s2[2 * I * H // 32:] += 1                  # every down scale doubled
    y2, h2 = oracle.expert_forward(codes, s2, H, I, x)
    assert np.array_equal(h1, h2) and np.array_equal(y2, 2 * y1)


def test_dense_k_equals_E_is_softmax_moe():
    E, H, I = 8, 64, 32
    pool = oracle.SyntheticPool(21, E, H, I)
    x = synth.tokens_bf16(0, 0, 2, H)
    Wr = synth.router_bf16(22, E, H)
    d = oracle.decode_layer(pool, x, Wr, E)
    xf = synth.bf16_bits_to_f64(x)
    logits = xf @ synth.bf16_bits_to_f64(Wr).T           # fp64 sum: fine for weights
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    y = np.zeros((2, H))
    for e in range(E):
        codes, scales = pool(e)
        (cg, sg), (cu, su), (cd, sd) = _split(codes, scales, H, I)
        g = xf @ _dequant(cg, sg, I, H).T
        u = xf @ _dequant(cu, su, I, H).T
        y += p[:, e:e + 1] * ((g / (1 + np.exp(-g)) * u) @ _dequant(cd, sd, H, I).T)
    assert np.allclose(d["y"], y, rtol=1e-10, atol=1e-10 * np.abs(y).max())


# ------------------------------------------------------------------- prefill


def test_sort_pairs_is_the_stable_expert_major_order():
    rng = np.random.default_rng(3)
    T, k, E = 37, 4, 11
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    perm, inv, offsets = oracle.sort_pairs(idx, E)
    pairs = sorted(range(T * k), key=lambda p: (idx[p // k, p % k], p))
    assert list(perm) == pairs
    assert sorted(perm) == list(range(T * k))
    assert all(inv[perm[r]] == r for r in range(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert all(idx[p // k, p % k] == e for p in seg)
    assert offsets[-1] == T * k


# --------------------------------------------------------------- stacked glue


def test_prescale_is_exact_power_of_two():
    x = synth.tokens_bf16(10, 0, 3, 1024)
    x[1] = synth.bf16_bits_from_f64(synth.bf16_bits_to_f64(x[1]) * 37.0)
    xh = oracle.prescale(x)
    for r in range(3):
        a, b = synth.bf16_bits_to_f64(x[r]), synth.bf16_bits_to_f64(xh[r])
        amax = np.abs(b).max()
        assert 4 <= amax < 8
        ratio = a[a != 0] / b[a != 0]
        assert np.all(ratio == ratio[0]) and math.log2(ratio[0]).is_integer()


# --------------------------------------------------------------- byte counts


def test_expert_record_size_matches_the_pages():
    facts = {ln.split()[0]: float(ln.split()[1]) for ln in _golden_lines("page_facts.txt")}
    E = facts["routed_experts_total"] / facts["moe_layers"]
    assert E == synth.FULL.E == 896
    per_expert = synth.expert_code_bytes(7168, 1600) + synth.expert_scale_bytes(7168, 1600)
    assert per_expert == 18_278_400
    assert synth.expert_code_bytes(1024, 512) + synth.expert_scale_bytes(1024, 512) == 835_584
    mib = per_expert / 2**20
    assert abs(mib - facts["expert_record_mib"]) / facts["expert_record_mib"] < 0.005
    per_token = facts["experts_selected_per_layer"] * facts["moe_layers"] * mib / 1000
    assert abs(per_token - facts["expert_data_per_token_gb"]) / facts["expert_data_per_token_gb"] < 0.01


def test_mxfp8_ambiguity_marks_only_near_decisions():
    v = np.zeros(64)
    v[0] = 300.0                      # block amax well inside [256, 512): X = 0 (clear)
    v[1] = 1.0625                     # exact midpoint of 1.0 and 1.125 -> ambiguous
    v[2] = 1.0625 * (1 + 1e-6)        # within eps of it -> ambiguous
    v[3] = 1.03                       # far from a midpoint -> clear
    v[32] = 511.99                    # block max just below 2^9 -> the exponent may go up
    v[33] = 3.0
    d = oracle.mxfp8_ambiguity(v, 1e-4 * np.abs(v))
    assert d[0] == 0.0 and d[3] == 0.0
    assert d[1] == 0.125 and d[2] == 0.125
    assert d[32] > 0.0                # scale alternative 2^1 changes 511.99 -> 512 vs 448
    q = oracle.quant_mxfp8(v)[2]
    assert q[3] == 1.0 and q[1] == 1.0  # midpoint rounds to even (1.0)


# ------------------------------------------- MXFP8 h of the tensor-core path
# The prefill path quantises h = silu(g) * u to MXFP8 before W_d.  The GPU holds g
# and u as fp32 sums of block-scaled MMA steps (K = 32 each), so near an E4M3
# rounding midpoint or a power-of-two block max either MXFP8 choice is correct.  The
# oracle bounds the GPU's error in h (orc_h_radius) and the output change the open
# choices can make (orc_mxfp8_ambiguity, orc_expert_ambiguity); the pins below fix
# those pieces against an independent composition, an fp32 emulation of the step
# model and brute force.


def _one_expert(codes, scales):
    return lambda e: (codes, scales)


def test_expert_mxfp8_h_matches_independent_composition():
    """orc_expert_forward with h_mode 1 = dense dequantised W_g, W_u (bit-field
    definition) -> SwiGLU -> MXFP8 of h (the pinned block rule) -> dense W_d."""
    H, I = 256, 128
    codes, scales = oracle.gen_expert(17, 3, H, I)
    (cg, sg), (cu, su), (cd, sd) = _split(codes, scales, H, I)
    Wg, Wu, Wd = _dequant(cg, sg, I, H), _dequant(cu, su, I, H), _dequant(cd, sd, H, I)
    xq = oracle.quant_rows_mxfp8(synth.bf16_bits_to_f64(synth.tokens_bf16(13, 0, 3, H)))
    y, h = oracle.expert_forward(codes, scales, H, I, xq, h_mode=1)
    for m in range(3):
        g, u = Wg @ xq[m], Wu @ xq[m]
        hq = oracle.quant_mxfp8(g / (1 + np.exp(-g)) * u)[2]
        assert np.array_equal(h[m], hq)
        assert np.allclose(y[m], Wd @ hq, rtol=1e-13, atol=1e-13 * np.abs(y[m]).max())
    y0, _ = oracle.expert_forward(codes, scales, H, I, xq, h_mode=0)
    assert not np.array_equal(y, y0)          # the quantisation step is really applied


def _round_f32(v, mode):
    """fp64 values rounded once to fp32: nearest-even, toward zero, up or down."""
    r = v.astype(np.float32)
    rd = r.astype(np.float64)
    if mode == "ru":
        r = np.where(rd < v, np.nextafter(r, np.float32(np.inf)), r)
    elif mode == "rd":
        r = np.where(rd > v, np.nextafter(r, np.float32(-np.inf)), r)
    elif mode == "rz":
        r = np.where(np.abs(rd) > np.abs(v), np.nextafter(r, np.float32(0)), r)
    return r


def _fp32_steps(W, x, mode):
    """The fp32 accumulation of the step model: the exact sums of each 32-column block
    (in order) added to an fp32 running sum, one rounding per step."""
    blocks = (W * x[None, :]).reshape(W.shape[0], -1, 32).sum(axis=2)   # exact in fp64
    acc = _round_f32(blocks[:, 0], mode)
    for t in range(1, blocks.shape[1]):
        acc = _round_f32(acc.astype(np.float64) + blocks[:, t], mode)
    return acc


@pytest.mark.parametrize("mode", ["rn", "rz", "ru", "rd"])
def test_h_radius_covers_fp32_step_accumulation(mode):
    """The radius covers the error of an fp32 h built under the step model with any of
    the four rounding modes (and an fp32 epilogue), and is not far above the error that
    directed rounding actually reaches: a widened model constant fails here."""
    H, I = 1024, 256
    codes, scales = oracle.gen_expert(31, 4, H, I)
    (cg, sg), (cu, su), _ = _split(codes, scales, H, I)
    Wg, Wu = _dequant(cg, sg, I, H), _dequant(cu, su, I, H)
    # MXFP8 rows (as on the GPU: their short block sums often add up exactly in fp32)
    # and rows of full fp32 precision (every step rounds)
    xq = np.concatenate([oracle.quant_rows_mxfp8(synth.bf16_bits_to_f64(synth.tokens_bf16(12, 0, 2, H))),
                         np.random.default_rng(12).standard_normal((2, H)).astype(np.float32).astype(np.float64)])
    h, r = oracle.h_radius(codes, scales, H, I, xq)
    ratios = []
    for m in range(4):
        g, u = Wg @ xq[m], Wu @ xq[m]
        assert np.allclose(h[m], g / (1 + np.exp(-g)) * u, rtol=1e-12, atol=1e-12 * np.abs(h[m]).max())
        g32, u32 = _fp32_steps(Wg, xq[m], mode), _fp32_steps(Wu, xq[m], mode)
        h32 = (g32 / (np.float32(1) + np.exp(-g32)) * u32).astype(np.float64)
        err = np.abs(h32 - h[m])
        assert np.all(err <= r[m]), float(np.max(err / r[m]))
        if m >= 2:
            ratios.append(err / r[m])
    if mode in ("ru", "rd"):
        assert np.median(np.concatenate(ratios)) > 0.04


def test_mxfp8_ambiguity_bounds_every_choice_in_the_radius():
    """Brute force: values drawn anywhere in [v - r, v + r] (and at the ends) quantise
    to within delta of the nominal MXFP8 value, elements with delta 0 never change, and
    delta is reached for many of the open elements."""
    rng = np.random.default_rng(5)
    n = 32 * 48
    v = rng.standard_normal(n) * np.exp2(rng.integers(-3, 3, size=n))
    # planted decisions: E4M3 midpoints, and block maxima at a power of two
    v[3] = 1.0625 * 2.0 ** -6
    v[40] = 2.0 ** 3
    v[96:128] *= 0.1                  # element 100 the clear max of its block, just below 2
    v[100] = -(2.0 ** 1) * (1 - 1e-7)
    r = np.abs(v) * 10.0 ** rng.uniform(-7, -2, size=n)
    r[100] = 1e-6
    d = oracle.mxfp8_ambiguity(v, r)
    q0 = oracle.quant_mxfp8(v)[2]
    worst = np.zeros(n)
    for trial in range(400):
        pick = rng.integers(0, 3, size=n)
        vv = np.where(pick == 0, v - r, np.where(pick == 1, v + r, v + rng.uniform(-1, 1, size=n) * r))
        dq = np.abs(oracle.quant_mxfp8(vv)[2] - q0)
        assert np.all(dq <= d)
        worst = np.maximum(worst, dq)
    assert np.all(worst[d == 0] == 0)
    openi = d > 0
    assert openi.sum() > 20 and d[3] > 0 and d[40] > 0 and d[100] > 0
    assert np.mean(worst[openi] == d[openi]) > 0.25


def test_expert_ambiguity_bounds_the_output_change():
    """Brute force on a tiny expert with a large step error (so that many decisions
    are open): every h inside the radius gives an output within the per-output
    ambiguity of the nominal MXFP8-h output."""
    H, I = 256, 128
    rel = 2.0 ** -12
    codes, scales = oracle.gen_expert(19, 2, H, I)
    _, _, (cd, sd) = _split(codes, scales, H, I)
    Wd = _dequant(cd, sd, H, I)
    xq = oracle.quant_rows_mxfp8(synth.bf16_bits_to_f64(synth.tokens_bf16(14, 0, 2, H)))
    h, r = oracle.h_radius(codes, scales, H, I, xq, rel)
    amb = oracle.pair_ambiguity(_one_expert(codes, scales), H, I, xq, np.zeros((2, 1), np.int32), rel)[:, 0]
    y, _ = oracle.expert_forward(codes, scales, H, I, xq, h_mode=1)
    rng = np.random.default_rng(6)
    for m in range(2):
        o0 = Wd @ oracle.quant_mxfp8(h[m])[2]
        assert np.allclose(o0, y[m], rtol=1e-13, atol=1e-13 * np.abs(o0).max())
        for trial in range(150):
            hh = h[m] + r[m] * rng.choice([-1.0, 1.0, 0.0], size=I) * rng.uniform(0.5, 1.0, size=I)
            dq = np.abs(Wd @ oracle.quant_mxfp8(hh)[2] - o0)
            assert np.all(dq <= amb[m] * (1 + 1e-12) + 1e-14 * np.abs(o0).max())
        assert np.mean(amb[m] > 0) > 0.5


# ------------------------------------------------------- MXFP4 activations
# The prefill variant with FP4 activations quantises x and h to MXFP4 (OCP MX v1.0:
# E2M1 elements, one E8M0 scale per 32, shared exponent floor(log2 amax) - 2).


def test_e2m1_encode_round_trip_midpoints_and_saturation():
    mags = [oracle.e2m1_value(c) for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(8):
        assert oracle.e2m1_encode(mags[c]) == c
        assert oracle.e2m1_encode(-mags[c]) == (c | 8)
    for c in range(7):                          # exact midpoints go to the even code
        mid = (mags[c] + mags[c + 1]) / 2
        assert oracle.e2m1_encode(mid) == (c if c % 2 == 0 else c + 1)
        eps = (mags[c + 1] - mags[c]) * 1e-9
        assert oracle.e2m1_encode(mid - eps) == c
        assert oracle.e2m1_encode(mid + eps) == c + 1
    for big in [6.0, 6.5, 7.0, 100.0, 1e300]:
        assert oracle.e2m1_encode(big) == 7 and oracle.e2m1_encode(-big) == 15


def test_e2m1_encode_is_the_nearest_value():
    rng = np.random.default_rng(9)
    mags = np.array([oracle.e2m1_value(c) for c in range(8)])
    for v in rng.uniform(-7, 7, size=2000):
        c = oracle.e2m1_encode(v)
        got = oracle.e2m1_value(c)
        assert abs(abs(got) - min(abs(v), 6.0)) == np.min(np.abs(mags - min(abs(v), 6.0)))
        assert math.copysign(1, got) == math.copysign(1, v)


def test_mxfp4_block_rule():
    v = np.zeros(96)
    v[0] = 1.0          # amax 1 -> X = 0 - 2 = -2 (byte 125); 1 * 4 = 4 exact
    v[1] = -0.3         # 0.3 * 4 = 1.2 -> 1.0 -> -0.25
    v[32] = 7.0         # amax 7 -> X = 2 - 2 = 0; 7 saturates to 6
    v[33] = 2.5         # tie between 2 and 3 -> 2 (even)
    codes, sb, deq = oracle.quant_mxfp4(v)
    assert list(sb) == [125, 127, 0]
    assert deq[0] == 1.0 and deq[1] == -0.25
    assert deq[32] == 6.0 and deq[33] == 2.0
    assert np.all(deq[64:] == 0) and np.all(codes[2:32] == 0)


def test_mxfp4_error_bound_on_bf16_inputs():
    # the block max lies in [4, 8) * 2^X; every element is within half a step of its
    # value, the step being 2^(X + e - 1) for element exponent e >= 0, 2^(X-1) below
    x = synth.bf16_bits_to_f64(synth.tokens_bf16(0, 0, 4, 1024)).ravel()
    _, sb, deq = oracle.quant_mxfp4(x)
    for b in range(0, x.size, 32):
        X = int(sb[b // 32]) - 127
        blk = x[b:b + 32]
        assert 4 <= np.max(np.abs(blk)) / 2.0 ** X < 8
        t = np.abs(blk) / 2.0 ** X
        step = np.where(t >= 1, 2.0 ** (np.floor(np.log2(np.maximum(t, 1))) - 1), 0.5) * 2.0 ** X
        small = t <= 6
        assert np.all(np.abs(deq[b:b + 32] - blk)[small] <= step[small] / 2)


def test_expert_mxfp4_h_matches_independent_composition():
    H, I = 256, 128
    codes, scales = oracle.gen_expert(23, 1, H, I)
    (cg, sg), (cu, su), (cd, sd) = _split(codes, scales, H, I)
    Wg, Wu, Wd = _dequant(cg, sg, I, H), _dequant(cu, su, I, H), _dequant(cd, sd, H, I)
    xq = oracle.quant_rows_mxfp4(synth.bf16_bits_to_f64(synth.tokens_bf16(15, 0, 3, H)))
    y, h = oracle.expert_forward(codes, scales, H, I, xq, h_mode=2)
    for m in range(3):
        g, u = Wg @ xq[m], Wu @ xq[m]
        hq = oracle.quant_mxfp4(g / (1 + np.exp(-g)) * u)[2]
        assert np.array_equal(h[m], hq)
        assert np.allclose(y[m], Wd @ hq, rtol=1e-13, atol=1e-13 * np.abs(y[m]).max())


def test_mxfp4_ambiguity_bounds_every_choice_in_the_radius():
    rng = np.random.default_rng(8)
    n = 32 * 48
    v = rng.standard_normal(n) * np.exp2(rng.integers(-3, 3, size=n))
    v[3] = 1.25 * 2.0 ** -3           # an E2M1 midpoint at the block's scale
    r = np.abs(v) * 10.0 ** rng.uniform(-4, -0.7, size=n)
    d = oracle.mx_ambiguity(v, r, 4)
    q0 = oracle.quant_mxfp4(v)[2]
    worst = np.zeros(n)
    for trial in range(400):
        pick = rng.integers(0, 3, size=n)
        vv = np.where(pick == 0, v - r, np.where(pick == 1, v + r, v + rng.uniform(-1, 1, size=n) * r))
        dq = np.abs(oracle.quant_mxfp4(vv)[2] - q0)
        assert np.all(dq <= d)
        worst = np.maximum(worst, dq)
    assert np.all(worst[d == 0] == 0)
    assert (d > 0).sum() > 20 and np.mean(worst[d > 0] == d[d > 0]) > 0.25
