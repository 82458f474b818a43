"""Failure detection without a GPU fault: a bounded device wait that runs out.

Every device wait of the library is bounded.  Here the test-support hook makes the
grid barrier of the single-token decode kernel wait for one arrival that never
comes, with the wait limit lowered to 20 ms.  The kernel must then record
MOE_ERR_TIMEOUT, drain its own copies, and return; the context stays usable and
the next call on the same workspace must give the normal result, bit for bit."""
import time

import numpy as np
import pytest
import torch

import synth
from tests._util import to_dev_bf16

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("mxfp4_routed_expert_topk_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()


@pytest.mark.parametrize("shape", ["tiny", "full"])
def test_grid_barrier_timeout_reports_and_recovers(shape):
    s = synth.TINY if shape == "tiny" else synth.FULL
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, synth.pool_seed(0))
    Wr = to_dev_bf16(synth.router_bf16(synth.router_seed(0), s.E, s.H))
    x = to_dev_bf16(synth.tokens_bf16(synth.TOKENS_SEED["full"], 3, 1, s.H))
    idx, w = moe.moe_route_topk(x, Wr, s.k)
    ws = moe.workspace(moe.moe_workspace_size(moe.MOE_OP_DECODE, s.E, s.H, s.I, 1, s.k))
    y_ref = moe.moe_expert_forward_decode(pool, x, idx, w, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_OK

    sentinel = torch.full((1, s.H), 7.0, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    moe.moe_debug_set_wait_limit(20_000_000)          # 20 ms
    moe.moe_debug_set_barrier_extra(1)
    try:
        t0 = time.perf_counter()
        moe.moe_expert_forward_decode(pool, x, idx, w, ws=ws, y=sentinel)
        st = moe.moe_check_status(ws)                  # synchronises the stream
        elapsed = time.perf_counter() - t0
    finally:
        moe.moe_debug_set_barrier_extra(0)
        moe.moe_debug_set_wait_limit(0)
    assert st == moe.MOE_ERR_TIMEOUT, moe.status_string(st)
    assert elapsed < 2.0                               # the short limit, not the 1 s default
    assert torch.all(sentinel.float() == 7.0)          # an aborted call writes no y

    # the same workspace, the default limit: the normal result, bit for bit
    y2 = moe.moe_expert_forward_decode(pool, x, idx, w, ws=ws)
    assert moe.moe_check_status(ws) == moe.MOE_OK
    assert torch.equal(y2.view(torch.int16), y_ref.view(torch.int16))
    assert np.isfinite(y2.float().cpu().numpy()).all()
