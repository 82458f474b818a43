"""The router entry point for callers that cannot allocate device memory.

moe_route_topk_static keeps its scratch in a static device array of the
library instead of a caller workspace (for callers that cannot call cudaMalloc
or supply one).  Called through the C ABI, it must give the same routing as
moe_route_topk, on consecutive calls that reuse the shared array.  This file is
collected last so that a run stopping at the first failure has run every other
test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests._util import to_dev_bf16

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("mxfp4_routed_expert_topk_gb300")


def _static_route(L, x, Wr, k, skew=None):
    M, H = x.shape
    E = Wr.shape[0]
    idx = torch.full((M, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((M, k), -1.0, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    sk = None if skew is None else ctypes.c_void_p(skew.data_ptr())
    rc = L.moe_route_topk_static(ctypes.c_void_p(x.data_ptr()), M, H, ctypes.c_void_p(Wr.data_ptr()), E, sk, k,
                                 ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(w.data_ptr()), stream)
    assert rc == moe.MOE_OK, moe.status_string(rc)
    return idx, w


def test_static_router_matches_workspace_router():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.build()
    L = moe.lib()
    s = synth.FULL
    Wr = to_dev_bf16(synth.router_bf16(synth.router_seed(0), s.E, s.H))
    skew = torch.from_numpy(synth.zipf_skew_f32(synth.skew_seed(0), s.E)).cuda()
    # calls in a row share the array: M = 17 and 5 (the few-token logit kernel), then
    # M = 1 (the single-kernel router with its ticket counter in the status word) and
    # M = 128 (the many-token tiled router, whose row norms also live in the array;
    # 128 x 896 = 114,688 <= 131,072)
    calls = [(synth.tokens_bf16(synth.TOKENS_SEED["full"], 0, 17, s.H), None),
             (synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 0, 5, s.H), skew),
             (synth.tokens_bf16(synth.TOKENS_SEED["full"], 40, 1, s.H), None),
             (synth.tokens_bf16(synth.TOKENS_SEED["full"], 41, 1, s.H), skew),
             (synth.tokens_bf16(synth.TOKENS_SEED["full"], 100, 128, s.H), None),
             (synth.tokens_bf16(synth.TOKENS_SEED["stacked"], 100, 128, s.H), skew)]
    for xb, sk in calls:
        x = to_dev_bf16(xb)
        idx_s, w_s = _static_route(L, x, Wr, s.k, sk)
        idx_r, w_r = moe.moe_route_topk(x, Wr, s.k, sk)
        torch.cuda.synchronize()
        assert torch.equal(idx_s, idx_r)
        # the routing tests' weight tolerance (the kernels are the same, so in
        # practice the weights agree exactly)
        assert float((w_s - w_r).abs().max()) < 2e-6
    # sizes beyond the static array are rejected with a clear error
    big = torch.zeros((147, s.H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((147, s.k), dtype=torch.int32, device="cuda")
    w = torch.empty((147, s.k), dtype=torch.float32, device="cuda")
    rc = L.moe_route_topk_static(ctypes.c_void_p(big.data_ptr()), 147, s.H, ctypes.c_void_p(Wr.data_ptr()), s.E,
                                 None, s.k, ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == moe.MOE_ERR_UNSUPPORTED_SHAPE
