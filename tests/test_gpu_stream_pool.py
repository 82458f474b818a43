"""GPU: the layer through a streamed expert pool (records in pinned host memory, an
HBM cache of fewer slots than experts) gives bit for bit the output of the resident
pool, for single tokens and for a verify batch, while the cache misses, hits and
evicts."""
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


@pytest.mark.parametrize("shape,slots,ntok", [("tiny", 32, 24), ("full", 40, 6)])
def test_streamed_decode_matches_resident(shape, slots, ntok):
    s = synth.TINY if shape == "tiny" else synth.FULL
    pool = moe.Pool(s.E, s.H, s.I)
    moe.moe_pool_fill_synthetic(pool, synth.pool_seed(3))
    rec = moe.moe_pool_record_bytes(s.H, s.I)
    hb = moe.HostBuffer(s.E * rec)
    host = hb.tensor
    host.copy_(pool.mem)
    torch.cuda.synchronize()
    sp = moe.StreamPool(host, s.E, s.H, s.I, slots)
    Wr = to_dev_bf16(synth.router_bf16(synth.router_seed(3), s.E, s.H))
    skew = torch.from_numpy(synth.zipf_skew_f32(synth.skew_seed(3), s.E)).cuda()
    for t in range(ntok):
        x = to_dev_bf16(synth.tokens_bf16(synth.TOKENS_SEED["stacked"], t, 1, s.H))
        idx, w = moe.moe_route_topk(x, Wr, s.k, skew)
        y_ref = moe.moe_expert_forward_decode(pool, x, idx, w)
        slot = torch.from_numpy(sp.map(idx.cpu().numpy())).cuda()
        y = moe.moe_expert_forward_decode(sp.cache, x, slot, w)
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), t
    # a verify batch (grouped tensor-core path) through the same cache
    xb = to_dev_bf16(synth.verify_batch_bf16(synth.TOKENS_SEED["verify"], 7, 2, s.H))
    idx, w = moe.moe_route_topk(xb, Wr, s.k, skew)
    y_ref = moe.moe_expert_forward_decode(pool, xb, idx, w)
    slot = torch.from_numpy(sp.map(idx.cpu().numpy())).cuda()
    y = moe.moe_expert_forward_decode(sp.cache, xb, slot, w)
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    hits, misses, nbytes = sp.stats()
    assert hits > 0 and misses > slots and nbytes == misses * rec   # it evicted and refetched


def test_host_alloc_near_gpu():
    """moe_host_alloc: page-rounded pinned memory that host and device both reach, on
    the GPU's own host NUMA node when the system reports one."""
    want = moe.moe_host_numa_node()
    nbytes = (64 << 20) + 3
    hb = moe.HostBuffer(nbytes)
    if want >= 0:
        assert hb.numa_node == want
    pat = torch.arange(nbytes, dtype=torch.int64).remainder_(251).to(torch.uint8)
    hb.tensor.copy_(pat)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d.copy_(hb.tensor, non_blocking=True)
    back = torch.empty(nbytes, dtype=torch.uint8)
    back.copy_(d)
    assert torch.equal(back, pat)
    hb.close()
    hb.close()  # a second close is a no-op
