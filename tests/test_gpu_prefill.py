"""GPU parity of the expert-major prefill path: bit-exact pair permutation and
expert offsets, MXFP8 activations quantised as the oracle does, per-pair expert
outputs of the grouped tensor-core GEMMs and the combined layer output within the
float tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._util import bf16_to_f64, check_close, to_dev_bf16

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("mxfp4_routed_expert_topk_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    oracle.build()


def _run(s, T, seed, sample=None, partial_dtype=0):
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, seed)
    Wrb = synth.router_bf16(seed + 1, s.E, s.H)
    xb = synth.tokens_bf16(seed + 2, 0, T, s.H)
    x = to_dev_bf16(xb)
    idx, w = moe.moe_route_topk(x, to_dev_bf16(Wrb), s.k)
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_GROUPED, s.E, s.H, s.I, T, s.k))
    out = moe.moe_expert_forward_grouped(pool, x, idx, partial_dtype=partial_dtype, ws=ws)
    y = moe.moe_combine(out["partial"], out["inv_perm"], w)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    ref = oracle.prefill_layer(oracle.SyntheticPool(seed, s.E, s.H, s.I), xb, Wrb, s.k, act_mode=1,
                               sample_tokens=sample)
    return out, y, ref, xb


@pytest.mark.parametrize("E,H,I,k,T", [(16, 256, 128, 4, 64), (24, 384, 192, 8, 96), (64, 1024, 512, 16, 128)])
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
    check_close(part.reshape(T, s.k, s.H), o_ref, "partial", amb=p_amb)
    check_close(bf16_to_f64(y), ref["y"], "y", amb=ref["y_amb"])


def test_prefill_multiple_column_tiles():
    # 64 experts, 2048 tokens x 16 slots: ~512 rows per expert, several column tiles
    s = synth.TINY
    out, y, ref, _ = _run(s, 2048, 600, sample=np.arange(0, 2048, 97))
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    check_close(bf16_to_f64(y)[ref["tokens"]], ref["y"], "y", amb=ref["y_amb"])


def test_prefill_bf16_partials(tmp_path):
    s = synth.Shape(E=16, H=256, I=128, k=4)
    out, y, ref, _ = _run(s, 64, 516, partial_dtype=1)
    check_close(bf16_to_f64(y), ref["y"], "y", amb=ref["y_amb"])


def test_prefill_full_size_sampled():
    s = synth.FULL
    T = 512
    out, y, ref, _ = _run(s, T, 700, sample=np.arange(0, T, 73))
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])
    check_close(bf16_to_f64(y)[ref["tokens"]], ref["y"], "y", amb=ref["y_amb"])


def test_prefill_deterministic_after_other_shapes():
    """Same inputs, same bits: run once, dirty the GPU with another shape, run again."""
    s = synth.Shape(E=64, H=1024, I=512, k=16)
    out1, y1, _, _ = _run(s, 128, 564, sample=np.array([0]))
    _run(synth.Shape(E=16, H=256, I=128, k=4), 64, 516, sample=np.array([0]))
    out2, y2, _, _ = _run(s, 128, 564, sample=np.array([0]))
    assert torch.equal(out1["partial"], out2["partial"])
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
