"""CPU checks of the C-ABI library: it loads without a GPU, exports every entry
point include/moe.h declares, and its host-side validation and size arithmetic
behave as documented (none of these calls reaches the GPU)."""
import ctypes
import os
import re

import pytest

import mxfp4_routed_expert_topk_gb300 as moe
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 18
    for n in names:
        assert hasattr(L, n), n
    assert sorted(moe.EXPORTED) == names


def test_pool_sizes():
    full = moe.moe_pool_record_bytes(7168, 1600)
    # 18,278,400 B of MXFP4 data + zero padding of W_d rows to 1664 elements
    # (243,712 B) + the scale bytes once more in tensor-core order: W_gu 56 K tiles x
    # 25 row tiles x 512 B, W_d 13 x 56 x 512 B
    data = synth.expert_code_bytes(7168, 1600) + synth.expert_scale_bytes(7168, 1600)
    assert data == 18_278_400
    assert full == data + 243_712 + 56 * 25 * 512 + 13 * 56 * 512 == 19_611_648
    # 835,584 B of data (no padding), 8 x 8 x 512 + 4 x 8 x 512 B of reordered scales
    assert moe.moe_pool_record_bytes(1024, 512) == 835_584 + 8 * 8 * 512 + 4 * 8 * 512
    assert moe.moe_pool_bytes(896, 7168, 1600) == 896 * full
    assert moe.moe_pool_bytes(896, 7100, 1600) == 0      # H not a multiple of 128
    assert moe.moe_pool_bytes(896, 7168, 1601) == 0


def test_workspace_sizes_and_errors(L):
    assert moe.moe_workspace_size(moe.MOE_OP_ROUTE, 896, 7168, 1600, 1, 16) > 256
    assert moe.moe_workspace_size(moe.MOE_OP_DECODE, 896, 7168, 1600, 17, 16) > 256
    assert moe.moe_workspace_size(moe.MOE_OP_GROUPED, 896, 7168, 1600, 512, 16) > 512 * 16 * 7168
    with pytest.raises(moe.MoeError) as e:
        moe.moe_workspace_size(moe.MOE_OP_DECODE, 896, 7168, 1600, 33, 16)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(moe.MoeError) as e:
        moe.moe_workspace_size(moe.MOE_OP_ROUTE, 8, 1024, 512, 1, 16)   # k > E
    assert e.value.code == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_size(7, 64, 1024, 512, 1, 16)


def test_host_validation_without_gpu(L):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)   # never dereferenced: validation fails first
    assert L.moe_route_topk(None, 1, 1024, fake, 64, None, 16, fake, fake, fake, 1 << 20, None) == 1
    assert L.moe_route_topk(fake, 1, 1024, fake, 64, None, 65, fake, fake, fake, 1 << 20, None) == 1
    assert L.moe_route_topk(fake, 1, 1004, fake, 64, None, 16, fake, fake, fake, 1 << 20, None) == 2
    assert L.moe_route_topk(fake, 1, 1024, fake, 64, None, 16, fake, fake, fake, 16, None) == 3
    h = vp()
    assert L.moe_pool_create(ctypes.byref(h), vp(1 << 20), 1 << 30, 64, 1024, 512) == 0
    assert L.moe_expert_forward_decode(h, fake, 33, fake, fake, 16, None, fake, fake, 1 << 30, None) == 2
    assert L.moe_expert_forward_decode(h, fake, 1, fake, fake, 16, None, fake, fake, 16, None) == 3
    assert L.moe_expert_forward_grouped(h, fake, 4, fake, 16, 0, fake, fake, fake, fake, 0, fake, 1 << 30,
                                        None) == 1   # act mode
    L.moe_pool_destroy(h)
    assert L.moe_pool_create(ctypes.byref(h), vp((1 << 20) + 8), 1 << 30, 64, 1024, 512) == 1   # alignment
    assert L.moe_pool_create(ctypes.byref(h), vp(1 << 20), 1000, 64, 1024, 512) == 1           # too small
    assert L.moe_combine(None, 0, fake, fake, 1, 16, 1024, None, fake, None) == 1
    # the grouped GEMMs' tile-shape switch: modes 0..2, anything else rejected; 2 restored
    assert L.moe_grouped_set_cta_pairs(3) == 1 and L.moe_grouped_set_cta_pairs(-1) == 1
    assert L.moe_grouped_set_cta_pairs(0) == 0 and L.moe_grouped_set_cta_pairs(2) == 0
    for code in range(8):
        assert moe.status_string(code) not in ("", "unknown status")
