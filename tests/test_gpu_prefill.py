"""GPU parity of the expert-major prefill path: bit-exact pair permutation and
expert offsets, MXFP8 activations quantised as the oracle does, per-pair expert
outputs of the grouped tensor-core GEMMs and the combined layer output within the
float tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._util import bf16_half_ulp, bf16_to_f64, check_close, dequant_mxfp4, split_expert, to_dev_bf16

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("mxfp4_routed_expert_topk_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    oracle.build()


def _run(s, T, seed, sample=None, partial_dtype=0, act_mode=1):
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, seed)
    Wrb = synth.router_bf16(seed + 1, s.E, s.H)
    xb = synth.tokens_bf16(seed + 2, 0, T, s.H)
    x = to_dev_bf16(xb)
    idx, w = moe.moe_route_topk(x, to_dev_bf16(Wrb), s.k)
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_GROUPED, s.E, s.H, s.I, T, s.k))
    out = moe.moe_expert_forward_grouped(pool, x, idx, act_mode=act_mode, partial_dtype=partial_dtype, ws=ws)
    y = moe.moe_combine(out["partial"], out["inv_perm"], w)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    ref = oracle.prefill_layer(oracle.SyntheticPool(seed, s.E, s.H, s.I), xb, Wrb, s.k, act_mode=act_mode,
                               sample_tokens=sample)
    out["ws"], out["pool"] = ws, pool
    return out, y, ref, xb


# (16, 384, 192, 4, 1024): 256 rows per expert on 192-column tiles (two column tiles per
# expert), with an odd number of 128-row A tiles in both GEMMs (3 and 3)
@pytest.mark.parametrize("E,H,I,k,T", [(16, 256, 128, 4, 64), (24, 384, 192, 8, 96), (64, 1024, 512, 16, 128),
                                       (16, 384, 192, 4, 1024)])
def test_prefill_small_shapes(E, H, I, k, T):
    s = synth.Shape(E=E, H=H, I=I, k=k)
    out, y, ref, xb = _run(s, T, 500 + E)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(out["inv_perm"].cpu().numpy(), ref["inv_perm"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    # per-pair (unweighted) expert outputs straight from the grouped GEMMs
    pool = oracle.SyntheticPool(500 + E, s.E, s.H, s.I)
    xq = oracle.quant_rows_mxfp8(synth.bf16_bits_to_f64(xb))
    o_ref = oracle.pair_outputs(pool, s.H, s.I, xq, ref["idx"], h_mode=1)
    part = out["partial"].float().cpu().numpy().astype(np.float64)[out["inv_perm"].cpu().numpy()]
    p_amb = oracle.pair_ambiguity(pool, s.H, s.I, xq, ref["idx"])
    check_close(part.reshape(T, s.k, s.H), o_ref, "prefill small shapes: per-pair outputs", amb=p_amb)
    check_close(bf16_to_f64(y), ref["y"], "prefill small shapes: y", amb=ref["y_amb"], bf16_at=bf16_to_f64(y))


def test_prefill_multiple_column_tiles():
    # 64 experts, 2048 tokens x 16 slots: ~512 rows per expert, several column tiles
    s = synth.TINY
    out, y, ref, _ = _run(s, 2048, 600, sample=np.arange(0, 2048, 97))
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    yg = bf16_to_f64(y)[ref["tokens"]]
    check_close(yg, ref["y"], "prefill tiny T=2048: y (sampled)", amb=ref["y_amb"], bf16_at=yg)


def test_prefill_bf16_partials(tmp_path):
    """bf16 partial outputs: each partial is one more stated bf16 rounding, so each
    output may also differ by sum_j w_j * (half-ulp of partial j)."""
    s = synth.Shape(E=16, H=256, I=128, k=4)
    T, seed = 64, 516
    out, y, ref, xb = _run(s, T, seed, partial_dtype=1)
    pool = oracle.SyntheticPool(seed, s.E, s.H, s.I)
    xq = oracle.quant_rows_mxfp8(synth.bf16_bits_to_f64(xb))
    o_ref = oracle.pair_outputs(pool, s.H, s.I, xq, ref["idx"], h_mode=1)
    part_round = np.einsum("tj,tjh->th", np.abs(ref["w"]), bf16_half_ulp(o_ref))
    yg = bf16_to_f64(y)
    check_close(yg, ref["y"], "prefill bf16 partials: y", amb=ref["y_amb"] + part_round, bf16_at=yg)


def test_prefill_full_size_all_tokens():
    """The full-size 512-token prefill: the pair permutation bit-exact and every
    token's output within the tolerance."""
    s = synth.FULL
    T = 512
    out, y, ref, _ = _run(s, T, 700)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(out["inv_perm"].cpu().numpy(), ref["inv_perm"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    yg = bf16_to_f64(y)
    check_close(yg, ref["y"], "config 4: prefill T=512, all tokens", amb=ref["y_amb"], bf16_at=yg)


def _h_decisions_and_down_sums(pool, s, T, xb, idx_np, out, ws, seed, tokens, label, act_mode=1):
    """Checks on the GPU's MXFP8 h (read back from the workspace) for the pairs of
    `tokens`:
      - every element equals the oracle's MXFP8(h), or differs only where the oracle's
        error model of the GPU's fp32 h leaves that decision open, and by no more than
        the open range allows;
      - the down GEMM's fp32 output of the GPU's own h is within the model's step
        bound of the exact product: 2^-23 * sum_t (|P_{t-1}| + |S_t|) over the
        32-element K steps in ascending order (this measures the tensor pipe's
        accumulation, the premise of the h model, on the hardware itself).
    Returns (elements compared, mismatches, elements the model leaves open)."""
    hq, hs = moe.moe_grouped_read_h(pool, T, s.k, out["offsets"], ws, act_mode=act_mode)
    hq, hs = hq.cpu(), hs.cpu().numpy()
    fmt = 8 if act_mode == 1 else 4
    e2m1 = np.array([oracle.e2m1_value(c) for c in range(16)])
    inv = out["inv_perm"].cpu().numpy()
    part = out["partial"].float().cpu().numpy()
    opool = oracle.SyntheticPool(seed, s.E, s.H, s.I)
    wd_cache = {}
    n = mism = nopen = 0
    worst_step = 0.0
    for t in tokens:
        xq = oracle.quant_rows(synth.bf16_bits_to_f64(xb[t:t + 1]), act_mode)
        for j in range(s.k):
            e, r = int(idx_np[t, j]), int(inv[t * s.k + j])
            codes, scales = opool(e)
            h, rad = oracle.h_radius(codes, scales, s.H, s.I, xq)
            d = oracle.mx_ambiguity(h[0], rad[0], fmt)
            q_or = (oracle.quant_mxfp8 if act_mode == 1 else oracle.quant_mxfp4)(h[0])[2]
            if act_mode == 1:
                vals = hq[r].view(torch.float8_e4m3fn).to(torch.float64).numpy()
            else:
                vals = e2m1[hq[r].numpy() & 15]
            q_gpu = vals * np.repeat(np.exp2(hs[r].astype(np.float64) - 127), 32)
            diff = np.abs(q_gpu - q_or)
            assert np.all(diff <= d), f"{label}: pair ({t},{j}) h outside the open decisions"
            n += diff.size
            mism += int(np.count_nonzero(diff))
            nopen += int(np.count_nonzero(d))
            if e not in wd_cache:
                _, _, (cd, sd) = split_expert(codes, scales, s.H, s.I)
                wd_cache = {e: dequant_mxfp4(cd, sd, s.H, s.I)}
            blocks = (wd_cache[e] * q_gpu[None, :]).reshape(s.H, s.I // 32, 32).sum(axis=2)   # exact
            P = np.cumsum(blocks, axis=1)
            prev = np.concatenate([np.zeros((s.H, 1)), P[:, :-1]], axis=1)
            bound = 2.0 ** -23 * (np.abs(prev) + np.abs(blocks)).sum(axis=1)
            err = np.abs(part[r].astype(np.float64) - P[:, -1])
            assert np.all(err <= bound), f"{label}: pair ({t},{j}) down sum outside the step bound"
            worst_step = max(worst_step, float(np.max(err / np.maximum(bound, 1e-300))))
    print(f"{label}: {mism} of {n} h elements differ from the oracle's MXFP8 choice, "
          f"{nopen} open under the model; worst down-sum error {worst_step:.3f} of the step bound")
    return n, mism, nopen


@pytest.mark.parametrize("shape,T,tokens", [("tiny", 128, None), ("full", 512, (0, 170, 341, 511))])
def test_prefill_h_decisions_follow_the_error_model(shape, T, tokens):
    s = synth.TINY if shape == "tiny" else synth.FULL
    seed = 910 + T
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, seed)
    xb = synth.tokens_bf16(seed + 2, 0, T, s.H)
    x = to_dev_bf16(xb)
    idx, w = moe.moe_route_topk(x, to_dev_bf16(synth.router_bf16(seed + 1, s.E, s.H)), s.k)
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_GROUPED, s.E, s.H, s.I, T, s.k))
    out = moe.moe_expert_forward_grouped(pool, x, idx, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    toks = range(T) if tokens is None else tokens
    n, mism, nopen = _h_decisions_and_down_sums(pool, s, T, xb, idx.cpu().numpy(), out, ws, seed, toks,
                                                f"h decisions {shape} T={T}")
    assert mism <= nopen


def test_prefill_deterministic_after_other_shapes():
    """Same inputs, same bits: run once, dirty the GPU with another shape, run again."""
    s = synth.Shape(E=64, H=1024, I=512, k=16)
    out1, y1, _, _ = _run(s, 128, 564, sample=np.array([0]))
    _run(synth.Shape(E=16, H=256, I=128, k=4), 64, 516, sample=np.array([0]))
    out2, y2, _, _ = _run(s, 128, 564, sample=np.array([0]))
    assert torch.equal(out1["partial"], out2["partial"])
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def _align(v, a):
    return (v + a - 1) // a * a


def _tensor_core_planes(rec, H, I):
    """The record's two scale planes in the tensor-core order, derived on the host from
    its row-major planes by the layout's definition: block (kt, mt) byte 16l + 4q + j =
    scale block 4kt + j of row 128mt + 32q + l, rows past the matrix 0."""
    Ip = _align(I, 128)
    gu_codes, d_codes = 2 * I * H // 2, H * Ip // 2
    off_sgu = gu_codes + d_codes
    off_sd = off_sgu + 2 * I * H // 32
    want = []
    for off, rows, nblk in ((off_sgu, 2 * I, H // 32), (off_sd, H, Ip // 32)):
        S = rec[off:off + rows * nblk].reshape(rows, nblk)
        nmt = -(-rows // 128)
        Sp = np.zeros((nmt * 128, nblk), dtype=np.uint8)
        Sp[:rows] = S
        # [mt][q][l][kt][j] -> [kt][mt][l][q][j]
        want.append(Sp.reshape(nmt, 4, 32, nblk // 4, 4).transpose(3, 0, 2, 1, 4).reshape(-1))
    off_sgu_mma = _align(off_sd + H * Ip // 32, 1024)
    off_sd_mma = off_sgu_mma + _align(want[0].size, 1024)
    got = [rec[off_sgu_mma:off_sgu_mma + want[0].size], rec[off_sd_mma:off_sd_mma + want[1].size]]
    return want, got, _align(off_sd_mma + want[1].size, 1024)


@pytest.mark.parametrize("H,I", [(256, 96), (384, 192), (1024, 512)])
def test_pool_tensor_core_scale_planes(H, I):
    """The derived scale planes hold exactly the row-major scale bytes, permuted, for a
    synthetic fill and for an uploaded expert (odd row-tile counts and padded W_d rows
    included)."""
    E = 3
    pool = moe.Pool(E, H, I)
    moe.moe_pool_fill_synthetic(pool, 41)
    g = torch.Generator().manual_seed(H + I)
    codes = torch.randint(0, 256, (3 * H * I // 2,), dtype=torch.uint8, generator=g).cuda()
    scales = torch.randint(0, 256, (3 * H * I // 32,), dtype=torch.uint8, generator=g).cuda()
    moe.moe_pool_upload_expert(pool, 1, codes, scales)
    torch.cuda.synchronize()
    rb = moe.moe_pool_record_bytes(H, I)
    mem = pool.mem.cpu().numpy()
    for e in range(E):
        want, got, rec_bytes = _tensor_core_planes(mem[e * rb:(e + 1) * rb], H, I)
        assert rec_bytes == rb
        for w_, g_ in zip(want, got):
            assert np.array_equal(w_, g_), e


def test_prefill_bad_index_sets_status():
    """Slots with an expert index out of range: the status word says so, those pairs are
    left out of the sort (inv_perm -1), and every other pair's output is still right."""
    s = synth.Shape(E=16, H=256, I=128, k=4)
    T, seed = 64, 531
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, seed)
    xb = synth.tokens_bf16(seed + 2, 0, T, s.H)
    x = to_dev_bf16(xb)
    idx, w = moe.moe_route_topk(x, to_dev_bf16(synth.router_bf16(seed + 1, s.E, s.H)), s.k)
    idx[5, 2] = 10_000
    idx[7, 0] = -3
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_GROUPED, s.E, s.H, s.I, T, s.k))
    out = moe.moe_expert_forward_grouped(pool, x, idx, ws=ws)
    y = moe.moe_combine(out["partial"], out["inv_perm"], w)
    assert moe.moe_check_status(ws) == moe.MOE_ERR_BAD_INDEX
    inv = out["inv_perm"].cpu().numpy().reshape(T, s.k)
    assert inv[5, 2] == -1 and inv[7, 0] == -1
    assert out["offsets"].cpu().numpy()[-1] == T * s.k - 2
    assert torch.isfinite(y.float()).all()
    idx_ok = idx.cpu().numpy().copy()
    idx_ok[5, 2] = 0
    idx_ok[7, 0] = 0
    opool = oracle.SyntheticPool(seed, s.E, s.H, s.I)
    xq = oracle.quant_rows_mxfp8(synth.bf16_bits_to_f64(xb))
    o_ref = oracle.pair_outputs(opool, s.H, s.I, xq, idx_ok, h_mode=1)
    amb = oracle.pair_ambiguity(opool, s.H, s.I, xq, idx_ok)
    valid = inv >= 0
    # rows past offsets[E] were never written: select the valid pairs' rows before casting
    part = out["partial"].float().cpu().numpy()[np.where(valid, inv, 0)].astype(np.float64)
    check_close(part[valid], o_ref[valid], "prefill bad index: per-pair outputs", amb=amb[valid])


@pytest.mark.parametrize("T,nsample", [(2048, 64), (8192, 64)])
def test_prefill_full_size_sweep_sampled(T, nsample):
    """The 2048- and 8192-token prefill at the full shape, in the launch configuration the
    benchmark times: exact routing of 64 sampled tokens, the pair permutation of the
    oracle's stable sort over all pairs, and the sampled tokens' outputs."""
    s = synth.FULL
    seed = 720 + T
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, seed)
    Wrb = synth.router_bf16(seed + 1, s.E, s.H)
    xb = synth.tokens_bf16(seed + 2, 0, T, s.H)
    x = to_dev_bf16(xb)
    idx, w = moe.moe_route_topk(x, to_dev_bf16(Wrb), s.k)
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_GROUPED, s.E, s.H, s.I, T, s.k))
    out = moe.moe_expert_forward_grouped(pool, x, idx, ws=ws)
    y = moe.moe_combine(out["partial"], out["inv_perm"], w)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    idx_g = idx.cpu().numpy()
    toks = np.linspace(0, T - 1, nsample).astype(np.int64)
    ridx, rw, _ = oracle.route(xb[toks], Wrb, s.k)
    assert np.array_equal(idx_g[toks], ridx)
    assert np.max(np.abs(w.cpu().numpy()[toks] - rw)) < 2e-6
    perm, inv, offsets = oracle.sort_pairs(idx_g, s.E)
    assert np.array_equal(out["perm"].cpu().numpy(), perm)
    assert np.array_equal(out["inv_perm"].cpu().numpy(), inv)
    assert np.array_equal(out["offsets"].cpu().numpy(), offsets)
    opool = oracle.SyntheticPool(seed, s.E, s.H, s.I)
    xq = oracle.quant_rows_mxfp8(synth.bf16_bits_to_f64(xb[toks]))
    yref = oracle.combine_rows(opool, s.H, s.I, xq, ridx, rw, h_mode=1)
    amb = oracle.combine_ambiguity(opool, s.H, s.I, xq, ridx, rw)
    yg = bf16_to_f64(y)[toks]
    check_close(yg, yref, f"config 4: prefill T={T}, 64 sampled tokens", amb=amb, bf16_at=yg)


@pytest.mark.parametrize("T", [1, 3])
def test_prefill_fewer_pairs_than_experts(T):
    """16 or 48 pairs over 64 experts: most experts have no rows (the union list, empty
    tiles and a grid smaller than the SM count)."""
    s = synth.TINY
    out, y, ref, xb = _run(s, T, 540 + T)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    yg = bf16_to_f64(y)
    check_close(yg, ref["y"], "prefill fewer pairs than experts: y", amb=ref["y_amb"], bf16_at=yg)


@pytest.mark.parametrize("E,H,I,k,T", [(16, 256, 128, 4, 64), (64, 1024, 512, 16, 96)])
def test_prefill_hot_expert_spans_column_tiles(E, H, I, k, T):
    """Planted routing: every token sends slot 0 to expert 0, so that expert has T rows
    while the tiles are sized for the mean (2 or 3 column tiles on the two-CTAs-per-SM
    shape); each pair's output must match the oracle's."""
    s = synth.Shape(E=E, H=H, I=I, k=k)
    seed = 860 + E
    pool = moe.Pool(E, H, I)
    moe.moe_pool_fill_synthetic(pool, seed)
    xb = synth.tokens_bf16(seed + 2, 0, T, H)
    rng = np.random.default_rng(seed)
    idx_h = np.stack([np.concatenate([[0], 1 + rng.choice(E - 1, k - 1, replace=False)]) for _ in range(T)])
    idx = torch.from_numpy(idx_h.astype(np.int32)).cuda()
    x = to_dev_bf16(xb)
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_GROUPED, E, H, I, T, k))
    out = moe.moe_expert_forward_grouped(pool, x, idx, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    perm, inv, offsets = oracle.sort_pairs(idx_h, E)
    assert np.array_equal(out["perm"].cpu().numpy(), perm)
    assert offsets[1] - offsets[0] == T
    opool = oracle.SyntheticPool(seed, E, H, I)
    xq = oracle.quant_rows_mxfp8(synth.bf16_bits_to_f64(xb))
    o_ref = oracle.pair_outputs(opool, H, I, xq, idx_h, h_mode=1)
    amb = oracle.pair_ambiguity(opool, H, I, xq, idx_h)
    part = out["partial"].float().cpu().numpy().astype(np.float64)[out["inv_perm"].cpu().numpy()]
    check_close(part.reshape(T, k, H), o_ref, "prefill hot expert: per-pair outputs", amb=amb)


# ------------------------------------------------------- MXFP4 activations
# act_mode MOE_ACT_MXFP4: x and h quantised to MXFP4 (the oracle applies the same
# step), contractions as kind::mxf4 MMAs (E2M1 x E2M1).


@pytest.mark.parametrize("E,H,I,k,T", [(16, 256, 128, 4, 64), (24, 384, 192, 8, 96), (64, 1024, 512, 16, 128),
                                       (16, 384, 192, 4, 1024)])
def test_prefill_mxfp4_small_shapes(E, H, I, k, T):
    s = synth.Shape(E=E, H=H, I=I, k=k)
    seed = 940 + E
    out, y, ref, xb = _run(s, T, seed, act_mode=2)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    pool = oracle.SyntheticPool(seed, s.E, s.H, s.I)
    xq = oracle.quant_rows_mxfp4(synth.bf16_bits_to_f64(xb))
    o_ref = oracle.pair_outputs(pool, s.H, s.I, xq, ref["idx"], h_mode=2)
    part = out["partial"].float().cpu().numpy().astype(np.float64)[out["inv_perm"].cpu().numpy()]
    p_amb = oracle.pair_ambiguity(pool, s.H, s.I, xq, ref["idx"], fmt=4)
    check_close(part.reshape(T, s.k, s.H), o_ref, "prefill MXFP4 small shapes: per-pair outputs", amb=p_amb)
    yg = bf16_to_f64(y)
    check_close(yg, ref["y"], "prefill MXFP4 small shapes: y", amb=ref["y_amb"], bf16_at=yg)


@pytest.mark.parametrize("shape,T,tokens", [("tiny", 128, None), ("full", 512, (0, 255, 511))])
def test_prefill_mxfp4_h_decisions_follow_the_error_model(shape, T, tokens):
    s = synth.TINY if shape == "tiny" else synth.FULL
    seed = 960 + T
    out, _, ref, xb = _run(s, T, seed, sample=np.array([0]), act_mode=2)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])    # so the routing is the oracle's
    toks = range(T) if tokens is None else tokens
    n, mism, nopen = _h_decisions_and_down_sums(out["pool"], s, T, xb, ref["idx"], out, out["ws"], seed, toks,
                                                f"MXFP4 h decisions {shape} T={T}", act_mode=2)
    assert mism <= nopen


@pytest.mark.parametrize("T,nsample", [(512, 32), (2048, 16), (8192, 16)])
def test_prefill_mxfp4_full_size(T, nsample):
    s = synth.FULL
    out, y, ref, _ = _run(s, T, 980 + T, sample=np.linspace(0, T - 1, nsample).astype(np.int64), act_mode=2)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    yg = bf16_to_f64(y)[ref["tokens"]]
    check_close(yg, ref["y"], f"config 4 MXFP4: prefill T={T}, {nsample} sampled tokens", amb=ref["y_amb"],
                bf16_at=yg)


# ------------------------------------------------------- paired-SM tiles
# moe_grouped_set_cta_pairs(CTA_PAIRS_ALWAYS): one-part tiles of 128+ columns on CTA
# pairs (tcgen05 cta_group::2, M = 256, each CTA half of the tile's activation rows)
# with MXFP4 rows too (the default pairs MXFP8 rows only).


@pytest.fixture
def cta_pairs():
    moe.moe_grouped_set_cta_pairs(moe.CTA_PAIRS_ALWAYS)
    try:
        yield
    finally:
        moe.moe_grouped_set_cta_pairs(moe.CTA_PAIRS_MXFP8)


@pytest.mark.parametrize("act_mode", [1, 2])
def test_prefill_cta_pairs_small_shape(cta_pairs, act_mode):
    # 192-column tiles, two per expert; 3 row tiles of A in both GEMMs, so each expert's
    # last pair has no second tile
    s = synth.Shape(E=16, H=384, I=192, k=4)
    T, seed = 1024, 1010 + act_mode
    out, y, ref, xb = _run(s, T, seed, act_mode=act_mode)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    pool = oracle.SyntheticPool(seed, s.E, s.H, s.I)
    xf = synth.bf16_bits_to_f64(xb)
    xq = oracle.quant_rows_mxfp8(xf) if act_mode == 1 else oracle.quant_rows_mxfp4(xf)
    o_ref = oracle.pair_outputs(pool, s.H, s.I, xq, ref["idx"], h_mode=act_mode)
    part = out["partial"].float().cpu().numpy().astype(np.float64)[out["inv_perm"].cpu().numpy()]
    p_amb = oracle.pair_ambiguity(pool, s.H, s.I, xq, ref["idx"], fmt=8 if act_mode == 1 else 4)
    check_close(part.reshape(T, s.k, s.H), o_ref, f"CTA pairs, act_mode {act_mode}: per-pair outputs", amb=p_amb)
    yg = bf16_to_f64(y)
    check_close(yg, ref["y"], f"CTA pairs, act_mode {act_mode}: y", amb=ref["y_amb"], bf16_at=yg)


def test_prefill_cta_pairs_multiple_column_tiles(cta_pairs):
    s = synth.TINY
    out, y, ref, _ = _run(s, 2048, 1020, sample=np.arange(0, 2048, 97))
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    yg = bf16_to_f64(y)[ref["tokens"]]
    check_close(yg, ref["y"], "CTA pairs: tiny T=2048, y (sampled)", amb=ref["y_amb"], bf16_at=yg)


@pytest.mark.parametrize("act_mode", [1, 2])
def test_prefill_cta_pairs_full_size(cta_pairs, act_mode):
    s = synth.FULL
    T = 8192
    out, y, ref, _ = _run(s, T, 1030 + act_mode, sample=np.linspace(0, T - 1, 8).astype(np.int64), act_mode=act_mode)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    yg = bf16_to_f64(y)[ref["tokens"]]
    check_close(yg, ref["y"], f"CTA pairs, act_mode {act_mode}: prefill T=8192, 8 sampled tokens",
                amb=ref["y_amb"], bf16_at=yg)
