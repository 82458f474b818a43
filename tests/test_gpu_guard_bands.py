"""GPU: no entry point writes outside the buffers it is given.

Every output and workspace of a call is carved out of a larger allocation whose margins
(4 KB on each side) hold a canary byte; after the call the margins must be intact.  The
calls cover each kernel family: the single-token router (with and without the fused
pre-scale), the few-token and the tiled many-token router, the static-scratch router,
the fused single-token decode, the multi-row (verify) decode on the tensor cores, the
expert-major prefill in both activation formats with both partial types, and the
combine."""
import numpy as np
import pytest
import torch

import synth
from tests._util import to_dev_bf16

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("mxfp4_routed_expert_topk_gb300")

CANARY = 0xA5
GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


class Guarded:
    """Tensors carved out of allocations with canary margins; check() asserts that
    every margin still holds the canary."""

    def __init__(self):
        self.bufs = []

    def tensor(self, shape, dtype, zero=True):
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        buf = torch.full((GUARD + nbytes + GUARD + 256,), CANARY, dtype=torch.uint8, device="cuda")
        off = GUARD + (-(buf.data_ptr() + GUARD)) % 256
        mid = buf[off:off + nbytes]
        mid.zero_() if zero else mid.fill_(0x3C)
        self.bufs.append((buf, off, nbytes))
        return mid.view(dtype).view(shape)

    def workspace(self, nbytes):
        return self.tensor((nbytes,), torch.uint8)

    def check(self, what):
        torch.cuda.synchronize()
        for buf, off, nbytes in self.bufs:
            lo = buf[:off]
            hi = buf[off + nbytes:]
            assert bool((lo == CANARY).all()), f"{what}: write below a buffer"
            assert bool((hi == CANARY).all()), f"{what}: write above a buffer"


def _router(s, seed):
    Wrb = synth.router_bf16(seed, s.E, s.H)
    return to_dev_bf16(Wrb)


@pytest.mark.parametrize("M", [1, 5, 128])
def test_router_writes_stay_inside(M):
    s = synth.TINY
    g = Guarded()
    Wr = _router(s, synth.router_seed(0))
    x = to_dev_bf16(synth.tokens_bf16(synth.TOKENS_SEED["tiny"], 0, M, s.H))
    idx = g.tensor((M, s.k), torch.int32, zero=False)
    w = g.tensor((M, s.k), torch.float32, zero=False)
    ws = g.workspace(moe.moe_workspace_size(moe.MOE_OP_ROUTE, s.E, s.H, s.I, M, s.k))
    moe.moe_route_topk(x, Wr, s.k, ws=ws, idx=idx, w=w)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    g.check(f"moe_route_topk M={M}")
    if M == 1:
        xhat = g.tensor((1, s.H), torch.bfloat16, zero=False)
        moe.moe_route_topk_prescaled(x, Wr, s.k, ws=ws, idx=idx, w=w, xhat=xhat)
        assert moe.moe_check_status(ws) == moe.MOE_OK
        g.check("moe_route_topk_prescaled M=1")
    idx2 = g.tensor((M, s.k), torch.int32, zero=False)
    w2 = g.tensor((M, s.k), torch.float32, zero=False)
    moe.moe_route_topk_static(x, Wr, s.k, idx=idx2, w=w2)
    torch.cuda.synchronize()
    assert torch.equal(idx2, idx)
    g.check(f"moe_route_topk_static M={M}")


@pytest.mark.parametrize("shape,M", [("tiny", 1), ("tiny", 5), ("full", 1), ("full", 2)])
def test_decode_writes_stay_inside(shape, M):
    s = synth.TINY if shape == "tiny" else synth.FULL
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, synth.pool_seed(0))
    Wr = _router(s, synth.router_seed(0))
    g = Guarded()
    xb = synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], 3, M, s.H)
    x = to_dev_bf16(xb)
    res = to_dev_bf16(synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 1, M, s.H))
    idx, w = moe.moe_route_topk(x, Wr, s.k)
    y = g.tensor((M, s.H), torch.bfloat16, zero=False)
    ws = g.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, M, s.k))
    moe.moe_expert_forward_decode(pool, x, idx, w, residual=res, ws=ws, y=y)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    g.check(f"moe_expert_forward_decode {shape} M={M}")
    # a second call on the same workspace (its counters were reset by the first)
    moe.moe_expert_forward_decode(pool, x, idx, w, ws=ws, y=y)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    g.check(f"moe_expert_forward_decode {shape} M={M}, second call")


@pytest.mark.parametrize("act_mode,partial_dtype,pairs", [(moe.MOE_ACT_MXFP8, moe.MOE_PARTIAL_F32, False),
                                                          (moe.MOE_ACT_MXFP8, moe.MOE_PARTIAL_BF16, False),
                                                          (moe.MOE_ACT_MXFP4, moe.MOE_PARTIAL_F32, False),
                                                          (moe.MOE_ACT_MXFP8, moe.MOE_PARTIAL_F32, True),
                                                          (moe.MOE_ACT_MXFP4, moe.MOE_PARTIAL_BF16, True)])
def test_grouped_and_combine_writes_stay_inside(act_mode, partial_dtype, pairs):
    # pairs: 192-column tiles on CTA pairs (16 experts, 1024 tokens x 4 slots)
    s = synth.Shape(E=16, H=384, I=192, k=4) if pairs else synth.TINY
    T = 1024 if pairs else 48
    if pairs:
        moe.moe_grouped_set_cta_pairs(moe.CTA_PAIRS_ALWAYS)
    try:
        _grouped_and_combine(s, T, act_mode, partial_dtype)
    finally:
        moe.moe_grouped_set_cta_pairs(moe.CTA_PAIRS_MXFP8)


def _grouped_and_combine(s, T, act_mode, partial_dtype):
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, synth.pool_seed(0))
    Wr = _router(s, synth.router_seed(0))
    x = to_dev_bf16(synth.tokens_bf16(synth.TOKENS_SEED["prefill"], 0, T, s.H))
    idx, w = moe.moe_route_topk(x, Wr, s.k)
    g = Guarded()
    pdt = torch.float32 if partial_dtype == moe.MOE_PARTIAL_F32 else torch.bfloat16
    out = {"perm": g.tensor((T * s.k,), torch.int32, zero=False),
           "inv_perm": g.tensor((T * s.k,), torch.int32, zero=False),
           "offsets": g.tensor((s.E + 1,), torch.int32, zero=False),
           "partial": g.tensor((T * s.k, s.H), pdt, zero=False)}
    ws = g.workspace(moe.moe_workspace_size(moe.MOE_OP_GROUPED, s.E, s.H, s.I, T, s.k))
    moe.moe_expert_forward_grouped(pool, x, idx, act_mode=act_mode, partial_dtype=partial_dtype, ws=ws, out=out)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    g.check(f"moe_expert_forward_grouped act_mode={act_mode} partial={partial_dtype}")
    y = g.tensor((T, s.H), torch.bfloat16, zero=False)
    moe.moe_combine(out["partial"], out["inv_perm"], w, y=y)
    g.check("moe_combine")
    assert torch.isfinite(y.float()).all()
