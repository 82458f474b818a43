"""GPU parity of the pool, the router and the decode/verify path against the
fp64 oracle: bit-exact bytes and routing indices, float tolerance on outputs."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._util import bf16_to_bits, bf16_to_f64, check_close, report_close, to_dev_bf16

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("mxfp4_routed_expert_topk_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    oracle.build()


def make_pool(shape, seed):
    pool = moe.Pool(shape.E, shape.H, shape.I)
    moe.moe_pool_fill_synthetic(pool, seed)
    return pool


@pytest.fixture(scope="module")
def tiny():
    s = synth.TINY
    pool = make_pool(s, synth.pool_seed(0))
    Wrb = synth.router_bf16(synth.router_seed(0), s.E, s.H)
    return s, pool, Wrb, to_dev_bf16(Wrb)


@pytest.fixture(scope="module")
def full():
    s = synth.FULL
    pool = make_pool(s, synth.pool_seed(0))
    Wrb = synth.router_bf16(synth.router_seed(0), s.E, s.H)
    return s, pool, Wrb, to_dev_bf16(Wrb)


# ------------------------------------------------------------------ pool


def test_generator_agreement_tiny(tiny):
    s, pool, _, _ = tiny
    for e in range(s.E):
        c, sc = moe.moe_pool_download_expert(pool, e)
        rc, rs = oracle.gen_expert(synth.pool_seed(0), e, s.H, s.I)
        assert np.array_equal(c.cpu().numpy(), rc), e
        assert np.array_equal(sc.cpu().numpy(), rs), e


def test_generator_agreement_full_sampled(full):
    s, pool, _, _ = full
    for e in (0, 1, 447, 895):
        c, sc = moe.moe_pool_download_expert(pool, e)
        rc, rs = oracle.gen_expert(synth.pool_seed(0), e, s.H, s.I)
        assert np.array_equal(c.cpu().numpy(), rc), e
        assert np.array_equal(sc.cpu().numpy(), rs), e


@pytest.mark.parametrize("H,I", [(1024, 512), (384, 96), (256, 160)])
def test_upload_download_roundtrip(H, I):
    pool = moe.Pool(3, H, I)
    rng = np.random.default_rng(H + I)
    for e in range(3):
        c = rng.integers(0, 256, size=3 * H * I // 2, dtype=np.uint8)
        sc = rng.integers(110, 130, size=3 * H * I // 32, dtype=np.uint8)
        moe.moe_pool_upload_expert(pool, e, torch.from_numpy(c).cuda(), torch.from_numpy(sc).cuda())
        c2, s2 = moe.moe_pool_download_expert(pool, e)
        assert np.array_equal(c2.cpu().numpy(), c) and np.array_equal(s2.cpu().numpy(), sc)


# ---------------------------------------------------------------- router


def _route_check(xb, Wrb, Wr, k, skew=None):
    x = to_dev_bf16(xb)
    sk = None if skew is None else torch.from_numpy(skew).cuda()
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, Wrb.shape[0], xb.shape[1], 32, xb.shape[0], k))
    idx, w = moe.moe_route_topk(x, Wr, k, sk, ws=ws)
    torch.cuda.synchronize()
    nfb = moe.exact_fallbacks(ws)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    ridx, rw, _ = oracle.route(xb, Wrb, k, skew)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.max(np.abs(w.cpu().numpy() - rw)) < 2e-6
    return nfb


def test_route_tiny_bit_exact(tiny):
    s, _, Wrb, Wr = tiny
    xb = synth.tokens_bf16(synth.TOKENS_SEED["tiny"], 0, 200, s.H)
    _route_check(xb, Wrb, Wr, s.k)


# M >= 64 takes the tiled logit kernel (longer summation tree, Cauchy-Schwarz bound);
# 130 rows leave a ragged last tile of 2 tokens
@pytest.mark.parametrize("M", [48, 130])
def test_route_full_bit_exact(full, M):
    s, _, Wrb, Wr = full
    xb = synth.tokens_bf16(synth.TOKENS_SEED["full"], 0, M, s.H)
    _route_check(xb, Wrb, Wr, s.k)


@pytest.mark.parametrize("M", [24, 70])
def test_route_with_zipf_skew(full, M):
    s, _, Wrb, Wr = full
    xb = synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 0, M, s.H)
    _route_check(xb, Wrb, Wr, s.k, synth.zipf_skew_f32(synth.skew_seed(0), s.E))


@pytest.mark.parametrize("M, skewed", [(1, False), (1, True), (17, False), (40, True)])
def test_route_bound_covers_error(full, M, skewed):
    """Fewer than 64 tokens: each fp32 logit and its bound (read from the workspace
    after the call) satisfy |logit - exact| <= bound against the oracle's exact
    logits, and the running bound stays far below the a-priori gamma_d * sum|x w|
    (d = 24 roundings at H = 7168, the bound these kernels used before)."""
    s, _, Wrb, Wr = full
    xb = synth.tokens_bf16(synth.TOKENS_SEED["full"], 200, M, s.H)
    skew = synth.zipf_skew_f32(synth.skew_seed(0), s.E) if skewed else None
    x = to_dev_bf16(xb)
    sk = None if skew is None else torch.from_numpy(skew).cuda()
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, 32, M, s.k))
    moe.moe_route_topk(x, Wr, s.k, sk, ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws) == moe.MOE_OK
    n = M * s.E
    raw = ws.cpu().numpy()
    off_b = 256 + (n * 4 + 255) // 256 * 256
    logit = np.frombuffer(raw[256:256 + 4 * n].tobytes(), np.float32).reshape(M, s.E).astype(np.float64)
    bound = np.frombuffer(raw[off_b:off_b + 4 * n].tobytes(), np.float32).reshape(M, s.E).astype(np.float64)
    _, _, exact = oracle.route(xb, Wrb, s.k, skew)
    err = np.abs(logit - exact)
    # the oracle's logits are the exact values rounded once to fp64
    assert np.all(err <= bound + 2.0 ** -52 * np.abs(exact)), float(np.max(err / bound))
    S = np.abs(synth.bf16_bits_to_f64(xb)) @ np.abs(synth.bf16_bits_to_f64(Wrb)).T
    if skew is not None:
        S = S + np.abs(skew.astype(np.float64))[None, :]
    apriori = 25 * 2.0 ** -24 * S
    assert np.mean(bound) < 0.25 * np.mean(apriori)


@pytest.mark.parametrize("k", [1, 2, 16, 32])
def test_route_k_values(tiny, k):
    s, _, Wrb, Wr = tiny
    xb = synth.tokens_bf16(5, 0, 40, s.H)
    _route_check(xb, Wrb, Wr, k)


@pytest.mark.parametrize("M", [16, 80])
def test_route_planted_ties_take_exact_path(tiny, M):
    s, _, Wrb0, _ = tiny
    Wrb = Wrb0.copy()
    xb = synth.tokens_bf16(7, 0, M, s.H)
    # exact duplicates (ties -> lower index), and one-ulp near ties of a strong row
    strong = synth.bf16_bits_from_f64(np.sign(synth.bf16_bits_to_f64(xb[0])) * 0.05)
    for e in (3, 20, 41):
        Wrb[e] = strong
    Wrb[9] = strong
    Wrb[9, 100] += 1
    Wrb[50] = Wrb[17]
    Wrb[63] = Wrb[17]
    nfb = _route_check(xb, Wrb, to_dev_bf16(Wrb), s.k)
    assert nfb > 0


@pytest.mark.parametrize("M", [1, 3])
def test_route_threshold_fallback(full, M):
    # The experts of the select CTA's last warp (e mod 256 in 224..255) get strongly
    # negative logits for token 0: the filter threshold (the smallest per-warp
    # runner-up) then sits among them and more than 512 keys pass it, so the
    # selection takes its round-by-round branch.  Token 0 of M=1 runs the
    # single-kernel router; M=3 repeats the token (the planted rows are identical,
    # so for other tokens they would form one 96-way exact tie).
    s, _, Wrb0, _ = full
    Wrb = Wrb0.copy()
    xb = np.repeat(synth.tokens_bf16(synth.TOKENS_SEED["full"], 100, 1, s.H), M, axis=0)
    neg = synth.bf16_bits_from_f64(-0.05 * np.sign(synth.bf16_bits_to_f64(xb[0])))
    for e in range(s.E):
        if (e % 256) // 32 == 7:
            Wrb[e] = neg
    _route_check(xb, Wrb, to_dev_bf16(Wrb), s.k)


@pytest.mark.parametrize("M", [8, 72])
def test_route_large_dynamic_range(tiny, M):
    s, _, Wrb0, _ = tiny
    rng = np.random.default_rng(11)
    xb = synth.bf16_bits_from_f64(rng.standard_normal((M, s.H)) * np.exp2(rng.integers(-60, 60, size=(M, s.H))))
    Wrb = synth.bf16_bits_from_f64(rng.standard_normal((s.E, s.H)) * np.exp2(rng.integers(-40, 30, size=(s.E, s.H))))
    _route_check(xb, Wrb, to_dev_bf16(Wrb), s.k)


# ---------------------------------------------------------------- decode


def _decode_check(s, pool, Wrb, Wr, xb, seed, residual=None, label="decode", opool=None):
    x = to_dev_bf16(xb)
    idx, w = moe.moe_route_topk(x, Wr, s.k)
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, xb.shape[0], s.k))
    res = None if residual is None else to_dev_bf16(residual)
    y = moe.moe_expert_forward_decode(pool, x, idx, w, residual=res, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    opool = oracle.SyntheticPool(seed, s.E, s.H, s.I) if opool is None else opool
    ref = oracle.decode_layer(opool, xb, Wrb, s.k, residual_bits=residual)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    yg = bf16_to_f64(y)
    return check_close(yg, ref["y"], label, bf16_at=yg)


def test_decode_tiny_single_tokens(tiny):
    s, pool, Wrb, Wr = tiny
    opool = oracle.SyntheticPool(synth.pool_seed(0), s.E, s.H, s.I, cache=s.E)
    for t in range(32):
        xb = synth.tokens_bf16(synth.TOKENS_SEED["tiny"], t, 1, s.H)
        _decode_check(s, pool, Wrb, Wr, xb, synth.pool_seed(0), label="config 0: tiny decode, 32 tokens",
                      opool=opool)


@pytest.mark.parametrize("M", [2, 5, 9, 17, 32])
def test_decode_verify_tiny(tiny, M):
    s, pool, Wrb, Wr = tiny
    xb = synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], M, M, s.H)
    _decode_check(s, pool, Wrb, Wr, xb, synth.pool_seed(0), label="verify tiny M=2..32")


def test_route_full_1000_tokens_one_at_a_time(full):
    """Config 1 as the benchmark runs it: each of the 1000 seeded tokens routed by its
    own single-token call; every index bit-exact against the oracle's exact routing."""
    s, _, Wrb, Wr = full
    n = 1000
    xb = synth.tokens_bf16(synth.TOKENS_SEED["full"], 0, n, s.H)
    x = to_dev_bf16(xb)
    idx = torch.empty((n, s.k), dtype=torch.int32, device="cuda")
    w = torch.empty((n, s.k), dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, 1, s.k))
    for t in range(n):
        moe.moe_route_topk(x[t:t + 1], Wr, s.k, ws=ws, idx=idx[t:t + 1], w=w[t:t + 1])
    torch.cuda.synchronize()
    assert moe.moe_check_status(ws) == moe.MOE_OK
    ridx, rw, _ = oracle.route(xb, Wrb, s.k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.max(np.abs(w.cpu().numpy() - rw)) < 2e-6


def test_decode_full_single_tokens(full):
    """Config 1: 64 of the benchmark's tokens through the single-token path (router and
    fused decode kernel, one call each), every output within the tolerance."""
    s, pool, Wrb, Wr = full
    opool = oracle.SyntheticPool(synth.pool_seed(0), s.E, s.H, s.I, cache=64)
    for t in range(0, 1000, 1000 // 64)[:64]:
        xb = synth.tokens_bf16(synth.TOKENS_SEED["full"], t, 1, s.H)
        _decode_check(s, pool, Wrb, Wr, xb, synth.pool_seed(0), label="config 1: full decode, 64 tokens",
                      opool=opool)


def test_decode_full_wide_dynamic_range(full):
    """A single token whose elements span 2^-40 .. 2^40 (the fused kernel stages the
    token as f16 scaled to its max, so the small elements fall below f16 range):
    routing bit-exact and the output within the tolerance."""
    s, pool, Wrb, Wr = full
    rng = np.random.default_rng(40)
    xf = rng.standard_normal((1, s.H)) * np.exp2(rng.uniform(-40, 40, size=(1, s.H)))
    xb = synth.bf16_bits_from_f64(xf)
    _decode_check(s, pool, Wrb, Wr, xb, synth.pool_seed(0), label="config 1: token with 2^+-40 range")


@pytest.mark.parametrize("M", [2, 5, 9, 17])
def test_decode_full_verify_batches(full, M):
    """Config 3 at the full shape: three seeded batches of M correlated rows each, every
    distinct selected expert read once and applied to all rows routed to it."""
    s, pool, Wrb, Wr = full
    opool = oracle.SyntheticPool(synth.pool_seed(0), s.E, s.H, s.I, cache=160)
    for b in range(3):
        xb = synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], b, M, s.H)
        _decode_check(s, pool, Wrb, Wr, xb, synth.pool_seed(0), label=f"config 3: verify M={M}, 3 batches",
                      opool=opool)


@pytest.mark.parametrize("M", [20, 32])
def test_decode_verify_hot_expert_spans_tiles(tiny, M):
    """Planted routing for a verify batch: every row sends slot 0 to expert 0, so that
    expert has M rows (more than the 16 pairs of one tile of the five-part path); each
    row's output must match the oracle's on the same indices and weights."""
    s, pool, _, _ = tiny
    rng = np.random.default_rng(M)
    xb = synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], 50 + M, M, s.H)
    idx_h = np.stack([np.concatenate([[0], 1 + rng.choice(s.E - 1, s.k - 1, replace=False)]) for _ in range(M)])
    w_h = rng.dirichlet(np.ones(s.k), size=M)
    idx = torch.from_numpy(idx_h.astype(np.int32)).cuda()
    w = torch.from_numpy(w_h.astype(np.float32)).cuda()
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, M, s.k))
    y = moe.moe_expert_forward_decode(pool, to_dev_bf16(xb), idx, w, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    opool = oracle.SyntheticPool(synth.pool_seed(0), s.E, s.H, s.I, cache=s.E)
    ref = oracle.combine_rows(opool, s.H, s.I, synth.bf16_bits_to_f64(xb), idx_h, w_h.astype(np.float32).astype(np.float64))
    yg = bf16_to_f64(y)
    check_close(yg, ref, "verify with a hot expert (M rows)", bf16_at=yg)


@pytest.mark.parametrize("M", [2, 5])
def test_decode_verify_repeated_index_within_bound(tiny, M):
    """A verify batch whose rows repeat an index: with an expert named at most
    ceil16(5 M) / 5 times in all (3 for M = 2, 6 for M = 5) the narrow GEMM stages
    hold all its rows, and every output matches the oracle on the same indices."""
    s, pool, _, _ = tiny
    rng = np.random.default_rng(100 + M)
    limit = ((5 * M + 15) // 16 * 16) // 5
    xb = synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], 70 + M, M, s.H)
    idx_h = np.stack([rng.choice(np.arange(1, s.E), s.k, replace=False) for _ in range(M)])
    # expert 0: twice in row 0, once in each other row, up to the limit
    idx_h[0, :2] = 0
    for m in range(1, min(M, limit - 1)):
        idx_h[m, 0] = 0
    assert (idx_h == 0).sum() <= limit
    w_h = rng.dirichlet(np.ones(s.k), size=M)
    idx = torch.from_numpy(idx_h.astype(np.int32)).cuda()
    w = torch.from_numpy(w_h.astype(np.float32)).cuda()
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, M, s.k))
    y = moe.moe_expert_forward_decode(pool, to_dev_bf16(xb), idx, w, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    opool = oracle.SyntheticPool(synth.pool_seed(0), s.E, s.H, s.I, cache=s.E)
    ref = oracle.combine_rows(opool, s.H, s.I, synth.bf16_bits_to_f64(xb), idx_h, w_h.astype(np.float32).astype(np.float64))
    yg = bf16_to_f64(y)
    check_close(yg, ref, "verify with a repeated index", bf16_at=yg)


def test_decode_verify_expert_named_too_often(tiny):
    """M = 2: an expert named 4 times (more than the 3 that 16 reserved B rows hold)
    is reported as MOE_ERR_BAD_INDEX (y is then not valid); the status word clears on
    the first check."""
    s, pool, _, _ = tiny
    M = 2
    xb = synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], 90, M, s.H)
    idx_h = np.stack([np.arange(s.k) + 1, np.arange(s.k) + 1 + s.k]).astype(np.int32)
    idx_h[0, :2] = 0
    idx_h[1, :2] = 0
    w = torch.full((M, s.k), 1.0 / s.k, dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, M, s.k))
    moe.moe_expert_forward_decode(pool, to_dev_bf16(xb), torch.from_numpy(idx_h).cuda(), w, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_ERR_BAD_INDEX
    assert moe.moe_check_status(ws) == moe.MOE_OK


@pytest.mark.parametrize("E,H,I,k,M", [(40, 384, 96, 8, 3), (20, 256, 160, 4, 7), (33, 640, 224, 32, 2)])
def test_decode_ragged_shapes(E, H, I, k, M):
    s = synth.Shape(E=E, H=H, I=I, k=k)
    pool = make_pool(s, 77)
    Wrb = synth.router_bf16(78, E, H)
    xb = synth.tokens_bf16(79, 0, M, H)
    _decode_check(s, pool, Wrb, to_dev_bf16(Wrb), xb, 77)


def test_decode_residual(tiny):
    s, pool, Wrb, Wr = tiny
    xb = synth.tokens_bf16(3, 0, 3, s.H)
    res = synth.tokens_bf16(4, 0, 3, s.H)
    _decode_check(s, pool, Wrb, Wr, xb, synth.pool_seed(0), residual=res)


def test_decode_deterministic(full):
    s, pool, Wrb, Wr = full
    x = to_dev_bf16(synth.verify_batch_bf16(1, 1, 9, s.H))
    idx, w = moe.moe_route_topk(x, Wr, s.k)
    y1 = moe.moe_expert_forward_decode(pool, x, idx, w)
    y2 = moe.moe_expert_forward_decode(pool, x, idx, w)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_zero_and_closed_form_experts():
    H, I, k = 256, 128, 4
    pool = moe.Pool(8, H, I)
    zc = torch.zeros(3 * H * I // 2, dtype=torch.uint8, device="cuda")
    ones = torch.full((3 * H * I // 2,), 0x22, dtype=torch.uint8, device="cuda")
    s127 = torch.full((3 * H * I // 32,), 127, dtype=torch.uint8, device="cuda")
    for e in range(4):
        moe.moe_pool_upload_expert(pool, e, zc, s127)
    for e in range(4, 8):
        moe.moe_pool_upload_expert(pool, e, ones, s127)
    xb = synth.bf16_bits_from_f64(synth.bf16_bits_to_f64(synth.tokens_bf16(9, 0, 1, H)) / 16)
    x = to_dev_bf16(xb)
    w = torch.full((1, k), 1.0 / k, dtype=torch.float32, device="cuda")
    y0 = moe.moe_expert_forward_decode(pool, x, torch.tensor([[0, 1, 2, 3]], dtype=torch.int32, device="cuda"), w)
    assert torch.count_nonzero(y0.float()) == 0
    y1 = moe.moe_expert_forward_decode(pool, x, torch.tensor([[4, 5, 6, 7]], dtype=torch.int32, device="cuda"), w)
    s_ = float(np.sum(synth.bf16_bits_to_f64(xb)))
    want = I * (s_ / (1 + np.exp(-s_)) * s_)
    check_close(bf16_to_f64(y1), np.full((1, H), want), "closed-form experts", bf16_at=bf16_to_f64(y1))


@pytest.mark.parametrize("M", [1, 3])
def test_bad_index_sets_status(tiny, M):
    # M = 1: the fused single-token kernel; M = 3: sort, gather and grouped GEMMs
    s, pool, _, _ = tiny
    x = to_dev_bf16(synth.tokens_bf16(0, 0, M, s.H))
    idx = torch.stack([torch.arange(s.k, dtype=torch.int32) + 5 * m for m in range(M)]).cuda()
    idx[0, 3] = 10_000
    idx[M - 1, 0] = -1
    w = torch.full((M, s.k), 1.0 / s.k, dtype=torch.float32, device="cuda")
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, M, s.k))
    y = moe.moe_expert_forward_decode(pool, x, idx, w, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_ERR_BAD_INDEX
    assert torch.isfinite(y.float()).all()
    assert moe.moe_check_status(ws) == moe.MOE_OK      # cleared by the first check


@pytest.mark.parametrize("M", [1, 3])
def test_route_prescaled_matches_prescale_then_route(full, M):
    """moe_route_topk_prescaled writes x_hat = moe_prescale(x) bit for bit and routes it
    exactly as moe_route_topk routes x_hat (M = 1 folds the pre-scale into the router)."""
    s, _, _, Wr = full
    rng = np.random.default_rng(M)
    xb = synth.bf16_bits_from_f64(synth.bf16_bits_to_f64(synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 0, M, s.H))
                                  * np.exp2(rng.integers(-20, 20, size=(M, 1))))
    x = to_dev_bf16(xb)
    skew = torch.from_numpy(synth.zipf_skew_f32(synth.skew_seed(0), s.E)).cuda()
    idx_p, w_p, xh_p = moe.moe_route_topk_prescaled(x, Wr, s.k, skew)
    xh = moe.moe_prescale(x)
    idx_r, w_r = moe.moe_route_topk(xh, Wr, s.k, skew)
    torch.cuda.synchronize()
    assert torch.equal(xh_p.view(torch.int16), xh.view(torch.int16))
    assert np.array_equal(bf16_to_bits(xh_p), np.stack([oracle.prescale(xb[m]) for m in range(M)]))
    assert torch.equal(idx_p, idx_r)
    assert torch.equal(w_p, w_r)


def test_route_prescaled_exact_path(tiny):
    """Planted ties after the pre-scale: the single-token router's exact fallback reads
    the pre-scaled token it staged, and the indices match the oracle's on x_hat."""
    s, _, Wrb0, _ = tiny
    Wrb = Wrb0.copy()
    xb = synth.bf16_bits_from_f64(synth.bf16_bits_to_f64(synth.tokens_bf16(7, 0, 1, s.H)) * 1024.0)
    Wrb[50] = Wrb[17]
    Wrb[63] = Wrb[17]
    strong = synth.bf16_bits_from_f64(np.sign(synth.bf16_bits_to_f64(xb[0])) * 0.05)
    for e in (3, 20, 41):
        Wrb[e] = strong
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, 32, 1, s.k))
    idx, w, xh = moe.moe_route_topk_prescaled(to_dev_bf16(xb), to_dev_bf16(Wrb), s.k, ws=ws)
    torch.cuda.synchronize()
    assert moe.exact_fallbacks(ws) > 0
    assert moe.moe_check_status(ws) == moe.MOE_OK
    xhb = oracle.prescale(xb[0])[None, :]
    assert np.array_equal(bf16_to_bits(xh), xhb)
    ridx, rw, _ = oracle.route(xhb, Wrb, s.k, None)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.max(np.abs(w.cpu().numpy() - rw)) < 2e-6


def test_stacked_layers_oracle_forced(tiny):
    """Per layer on the oracle's own layer input: pre-scale bit-exact, routing bit-exact,
    layer output within tolerance."""
    s = synth.TINY
    L = 4
    pools = [oracle.SyntheticPool(synth.pool_seed(l), s.E, s.H, s.I) for l in range(L)]
    gpools = [make_pool(s, synth.pool_seed(l)) for l in range(L)]
    routers = [synth.router_bf16(synth.router_seed(l), s.E, s.H) for l in range(L)]
    skews = [synth.zipf_skew_f32(synth.skew_seed(l), s.E) for l in range(L)]
    xb = synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 0, 1, s.H)
    layers, _ = oracle.stacked_step(pools, routers, skews, xb, s.k)
    for l, ly in enumerate(layers):
        x = to_dev_bf16(ly["x"])
        xh = moe.moe_prescale(x)
        assert np.array_equal(bf16_to_bits(xh), ly["x_hat"])
        idx, w = moe.moe_route_topk(xh, to_dev_bf16(routers[l]), s.k, torch.from_numpy(skews[l]).cuda())
        assert np.array_equal(idx.cpu().numpy(), ly["idx"])
        y = moe.moe_expert_forward_decode(gpools[l], xh, idx, w, residual=x)
        # the layer output is bf16(x + MoE(x_hat)): its MoE part against the oracle's,
        # with the half-ulp of the bf16 residual stream; relative L1 on the output
        xl, xn = synth.bf16_bits_to_f64(ly["x"]), bf16_to_f64(y)
        check_close(xn - xl, ly["y"], "stacked tiny, oracle-forced", bf16_at=xn, l1_on=(xn, xl + ly["y"]))


def test_stacked_layers_full_size():
    """Config 2 at the full shape: 8 layers (each its own pool, router and Zipf skew),
    16 tokens, run on the GPU as the benchmark runs it (pre-scale folded into the
    single-token router, residual fused into the decode kernel).
      - Teacher-forced, per layer, on the GPU's own layer input x_l: the pre-scale
        bit-exact, the routing bit-exact and the MoE part of x_{l+1} = bf16(x_l +
        MoE(x_hat_l)) within the tolerance (plus the half-ulp of that bf16 rounding).
      - Free-running: the oracle's own 8-layer pass from the same x_0, each side
        feeding its own bf16 residual stream forward.  The two streams differ by
        one-ulp bf16 roundings from layer 1 on, and those move the logits by about
        3e-3 against a typical gap of about 0.04 between the 16th and 17th, so the
        routing of a token eventually diverges.  Per token the first layer whose
        routing differs is reported, and the streams entering it (x_8 if none) are
        compared: max|err|/RMS recorded, relative L1 held to the streams' own rounding,
        8 x 2^-9 (a bf16 half-ulp per layer)."""
    s = synth.FULL
    L, ntok = 8, 16
    pools = [make_pool(s, synth.pool_seed(l)) for l in range(L)]
    opools = [oracle.SyntheticPool(synth.pool_seed(l), s.E, s.H, s.I, cache=16) for l in range(L)]
    routers = [synth.router_bf16(synth.router_seed(l), s.E, s.H) for l in range(L)]
    skews = [synth.zipf_skew_f32(synth.skew_seed(l), s.E) for l in range(L)]
    Wrs = [to_dev_bf16(r) for r in routers]
    sks = [torch.from_numpy(k_).cuda() for k_ in skews]
    x0 = synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 0, ntok, s.H)
    ws_r = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, 1, s.k))
    ws_d = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, 1, s.k))
    # GPU pass: per token, per layer (x_l, x_hat_l, idx_l) kept for the checks
    xs = np.zeros((L + 1, ntok, s.H), dtype=np.uint16)
    xhs = np.zeros((L, ntok, s.H), dtype=np.uint16)
    idxs = np.zeros((L, ntok, s.k), dtype=np.int32)
    xs[0] = x0
    for t in range(ntok):
        x = to_dev_bf16(x0[t:t + 1])
        for l in range(L):
            idx, w, xh = moe.moe_route_topk_prescaled(x, Wrs[l], s.k, sks[l], ws=ws_r)
            y = moe.moe_expert_forward_decode(pools[l], xh, idx, w, residual=x, ws=ws_d)
            xhs[l, t], idxs[l, t] = bf16_to_bits(xh)[0], idx.cpu().numpy()[0]
            xs[l + 1, t] = bf16_to_bits(y)[0]
            x = y
    assert moe.moe_check_status(ws_r) == moe.MOE_OK and moe.moe_check_status(ws_d) == moe.MOE_OK
    # teacher-forced
    for l in range(L):
        xh_ref = oracle.prescale(xs[l])
        assert np.array_equal(xhs[l], xh_ref), l
        d = oracle.decode_layer(opools[l], xh_ref, routers[l], s.k, skews[l])
        assert np.array_equal(idxs[l], d["idx"]), l
        # x_{l+1} = bf16(x_l + MoE(x_hat_l)): the MoE part against the oracle's, with the
        # half-ulp of the bf16 residual stream; relative L1 on x_{l+1}
        xn, xl = synth.bf16_bits_to_f64(xs[l + 1]), synth.bf16_bits_to_f64(xs[l])
        check_close(xn - xl, d["y"], "config 2: 8 full layers, teacher-forced per layer", bf16_at=xn,
                    l1_on=(xn, xl + d["y"]))
    # free-running: each token until the first layer whose routing differs (or to the
    # end); the streams entering that layer are compared
    first, ys, refs = [], [], []
    for t in range(ntok):
        layers, x_fin = oracle.stacked_step(opools, routers, skews, x0[t], s.k)
        f = next((l for l, ly in enumerate(layers) if not np.array_equal(ly["idx"][0], idxs[l, t])), L)
        first.append(f)
        ys.append(synth.bf16_bits_to_f64(xs[f, t]))
        refs.append(synth.bf16_bits_to_f64(layers[f]["x"][0] if f < L else x_fin[0]))
    print(f"config 2 free-running: first layer whose routing diverged, per token (8 = none): {first}")
    # each side rounds its own stream to bf16 after every layer: at most a half-ulp
    # (2^-9 relative) per layer apart, over at most 8 layers
    report_close(np.stack(ys), np.stack(refs), "config 2: free-running stream at first divergence",
                 rel_l1=L * 2.0 ** -9)
    assert min(first) >= 1          # layer 0 sees the same x_0 on both sides
    del pools
    torch.cuda.empty_cache()


@pytest.mark.parametrize("E,H,M,k", [(100, 512, 70, 8), (1100, 256, 64, 16), (33, 384, 65, 4)])
def test_route_tiled_ragged_shapes(E, H, M, k):
    """The many-token logit kernel with expert counts that leave a partial 64-expert tile
    (and, for E > 1024, the selection with 8 keys per thread), bit-exact indices."""
    rng = np.random.default_rng(E + H + M)
    Wrb = synth.bf16_bits_from_f64(rng.standard_normal((E, H)) / np.sqrt(H))
    xb = synth.bf16_bits_from_f64(rng.standard_normal((M, H)))
    _route_check(xb, Wrb, to_dev_bf16(Wrb), k)
