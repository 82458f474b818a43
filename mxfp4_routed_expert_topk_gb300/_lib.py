"""ctypes binding of libmoe.so: argument marshalling only.

Every function here forwards to the entry point of the same name in
include/moe.h.  Tensors are PyTorch CUDA tensors (device memory and streams
come from PyTorch); all computation happens in the library's CUDA kernels.  If
the library has not been built the first call raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_BAD_INDEX = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_NONFINITE = 7

MOE_OP_ROUTE, MOE_OP_DECODE, MOE_OP_GROUPED = 0, 1, 2
MOE_ACT_MXFP8, MOE_ACT_MXFP4 = 1, 2
MOE_PARTIAL_F32, MOE_PARTIAL_BF16 = 0, 1

EXPORTED = [
    "moe_pool_bytes", "moe_pool_record_bytes", "moe_pool_create", "moe_pool_destroy",
    "moe_pool_fill_synthetic", "moe_pool_upload_expert", "moe_pool_download_expert",
    "moe_workspace_size", "moe_clear_status", "moe_check_status", "moe_status_string",
    "moe_route_topk", "moe_route_topk_static", "moe_route_topk_prescaled", "moe_expert_forward_decode",
    "moe_prescale",
    "moe_expert_forward_grouped", "moe_grouped_read_h", "moe_combine", "moe_grouped_set_cta_pairs",
    "moe_trace_begin", "moe_trace_end",
    "moe_debug_set_wait_limit", "moe_debug_set_barrier_extra",
    "moe_stream_pool_create", "moe_stream_pool_destroy", "moe_stream_pool_cache", "moe_stream_pool_slots",
    "moe_stream_pool_map", "moe_stream_pool_stats", "moe_host_alloc", "moe_host_free", "moe_host_numa_node",
]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


_lib = None
_vp, _sz, _i, _u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "moe_pool_bytes": (_sz, [_i, _i, _i]),
            "moe_pool_record_bytes": (_sz, [_i, _i]),
            "moe_pool_create": (_i, [ctypes.POINTER(_vp), _vp, _sz, _i, _i, _i]),
            "moe_pool_destroy": (None, [_vp]),
            "moe_pool_fill_synthetic": (_i, [_vp, _u64, _i, _i, _vp]),
            "moe_pool_upload_expert": (_i, [_vp, _i, _vp, _vp, _vp]),
            "moe_pool_download_expert": (_i, [_vp, _i, _vp, _vp, _vp]),
            "moe_workspace_size": (_i, [_i, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
            "moe_clear_status": (_i, [_vp, _vp]),
            "moe_check_status": (_i, [_vp, _vp]),
            "moe_status_string": (ctypes.c_char_p, [_i]),
            "moe_route_topk": (_i, [_vp, _i, _i, _vp, _i, _vp, _i, _vp, _vp, _vp, _sz, _vp]),
            "moe_route_topk_static": (_i, [_vp, _i, _i, _vp, _i, _vp, _i, _vp, _vp, _vp]),
            "moe_route_topk_prescaled": (_i, [_vp, _i, _i, _vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
            "moe_expert_forward_decode": (_i, [_vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp]),
            "moe_prescale": (_i, [_vp, _i, _i, _vp, _vp]),
            "moe_expert_forward_grouped": (_i, [_vp, _vp, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _sz,
                                                _vp]),
            "moe_grouped_read_h": (_i, [_vp, _i, _i, _i, _vp, _vp, _sz, _vp, _vp, _vp]),
            "moe_combine": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _vp]),
            "moe_debug_set_wait_limit": (_i, [_u64]),
            "moe_stream_pool_create": (_i, [ctypes.POINTER(_vp), _vp, _sz, _i, _i, _i, _vp, _sz]),
            "moe_stream_pool_destroy": (None, [_vp]),
            "moe_stream_pool_cache": (_vp, [_vp]),
            "moe_stream_pool_slots": (_i, [_vp]),
            "moe_stream_pool_map": (_i, [_vp, _vp, _i, _vp, _vp]),
            "moe_stream_pool_stats": (_i, [_vp, ctypes.POINTER(_u64), ctypes.POINTER(_u64), ctypes.POINTER(_u64)]),
            "moe_host_alloc": (_i, [_i, _sz, ctypes.POINTER(_vp), ctypes.POINTER(_i)]),
            "moe_host_free": (_i, [_vp, _sz]),
            "moe_host_numa_node": (_i, [_i]),
            "moe_debug_set_barrier_extra": (_i, [_i]),
            "moe_grouped_set_cta_pairs": (_i, [_i]),
            "moe_trace_begin": (_i, [ctypes.c_char_p]),
            "moe_trace_end": (_i, [ctypes.POINTER(_i), ctypes.POINTER(ctypes.c_double)]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoeError(code, where)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor")


# ------------------------------------------------------------------ pool


def moe_pool_bytes(E: int, H: int, I: int) -> int:
    return int(lib().moe_pool_bytes(E, H, I))


def moe_pool_record_bytes(H: int, I: int) -> int:
    return int(lib().moe_pool_record_bytes(H, I))


class Pool:
    """A resident expert pool in a caller-owned (PyTorch) device buffer."""

    def __init__(self, E: int, H: int, I: int, device="cuda", buffer: torch.Tensor | None = None):
        self.E, self.H, self.I = E, H, I
        nbytes = moe_pool_bytes(E, H, I)
        if nbytes == 0:
            raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_pool_bytes")
        if buffer is None:
            buffer = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device)
        self.buffer = buffer
        off = (-buffer.data_ptr()) % 1024
        self.mem = buffer[off:off + nbytes]
        h = ctypes.c_void_p()
        _check(lib().moe_pool_create(ctypes.byref(h), _ptr(self.mem), nbytes, E, H, I), "moe_pool_create")
        self.handle = h

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.moe_pool_destroy(h)
            self.handle = None


def moe_pool_fill_synthetic(pool: Pool, seed: int, e_lo: int = 0, e_hi: int | None = None, stream=None):
    e_hi = pool.E if e_hi is None else e_hi
    _check(lib().moe_pool_fill_synthetic(pool.handle, seed, e_lo, e_hi, _stream(stream)),
           "moe_pool_fill_synthetic")


def moe_pool_upload_expert(pool: Pool, e: int, codes: torch.Tensor, scales: torch.Tensor, stream=None):
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.uint8, "scales")
    _check(lib().moe_pool_upload_expert(pool.handle, e, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_pool_upload_expert")


def moe_pool_download_expert(pool: Pool, e: int, stream=None):
    codes = torch.empty(3 * pool.H * pool.I // 2, dtype=torch.uint8, device=pool.mem.device)
    scales = torch.empty(3 * pool.H * pool.I // 32, dtype=torch.uint8, device=pool.mem.device)
    _check(lib().moe_pool_download_expert(pool.handle, e, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_pool_download_expert")
    return codes, scales


# ------------------------------------------------------------- workspace


def moe_workspace_size(op: int, E: int, H: int, I: int, rows: int, k: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_workspace_size(op, E, H, I, rows, k, ctypes.byref(n)), "moe_workspace_size")
    return int(n.value)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace buffer (status word cleared), 256-byte aligned."""
    buf = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + nbytes]


def moe_clear_status(ws: torch.Tensor, stream=None):
    _check(lib().moe_clear_status(_ptr(ws), _stream(stream)), "moe_clear_status")


def moe_check_status(ws: torch.Tensor, stream=None) -> int:
    return int(lib().moe_check_status(_ptr(ws), _stream(stream)))


def exact_fallbacks(ws: torch.Tensor) -> int:
    """Router diagnostic: tokens that needed exact re-evaluation (status word slot 2)."""
    return int(ws[8:12].view(torch.int32).item())


# ---------------------------------------------------------------- layer


def moe_route_topk(x: torch.Tensor, Wr: torch.Tensor, k: int, skew: torch.Tensor | None = None,
                   ws: torch.Tensor | None = None, idx: torch.Tensor | None = None,
                   w: torch.Tensor | None = None, stream=None):
    _need(x, torch.bfloat16, "x")
    _need(Wr, torch.bfloat16, "Wr")
    M, H = x.shape
    E = Wr.shape[0]
    if skew is not None:
        _need(skew, torch.float32, "skew")
    if ws is None:
        ws = workspace(moe_workspace_size(MOE_OP_ROUTE, E, H, 32, M, k), x.device)
    idx = torch.empty((M, k), dtype=torch.int32, device=x.device) if idx is None else idx
    w = torch.empty((M, k), dtype=torch.float32, device=x.device) if w is None else w
    _check(lib().moe_route_topk(_ptr(x), M, H, _ptr(Wr), E, _ptr(skew), k, _ptr(idx), _ptr(w), _ptr(ws),
                                ws.numel(), _stream(stream)), "moe_route_topk")
    return idx, w


def moe_route_topk_prescaled(x: torch.Tensor, Wr: torch.Tensor, k: int, skew: torch.Tensor | None = None,
                             ws: torch.Tensor | None = None, idx: torch.Tensor | None = None,
                             w: torch.Tensor | None = None, xhat: torch.Tensor | None = None, stream=None):
    """Route x_hat = moe_prescale(x); returns (idx, w, x_hat)."""
    _need(x, torch.bfloat16, "x")
    _need(Wr, torch.bfloat16, "Wr")
    M, H = x.shape
    E = Wr.shape[0]
    if skew is not None:
        _need(skew, torch.float32, "skew")
    if ws is None:
        ws = workspace(moe_workspace_size(MOE_OP_ROUTE, E, H, 32, M, k), x.device)
    idx = torch.empty((M, k), dtype=torch.int32, device=x.device) if idx is None else idx
    w = torch.empty((M, k), dtype=torch.float32, device=x.device) if w is None else w
    xhat = torch.empty_like(x) if xhat is None else xhat
    _need(xhat, torch.bfloat16, "xhat")
    _check(lib().moe_route_topk_prescaled(_ptr(x), M, H, _ptr(Wr), E, _ptr(skew), k, _ptr(idx), _ptr(w), _ptr(xhat),
                                          _ptr(ws), ws.numel(), _stream(stream)), "moe_route_topk_prescaled")
    return idx, w, xhat


def moe_route_topk_static(x: torch.Tensor, Wr: torch.Tensor, k: int, skew: torch.Tensor | None = None,
                          idx: torch.Tensor | None = None, w: torch.Tensor | None = None, stream=None):
    """moe_route_topk without a workspace (the library's static scratch array)."""
    _need(x, torch.bfloat16, "x")
    _need(Wr, torch.bfloat16, "Wr")
    M, H = x.shape
    E = Wr.shape[0]
    idx = torch.empty((M, k), dtype=torch.int32, device=x.device) if idx is None else idx
    w = torch.empty((M, k), dtype=torch.float32, device=x.device) if w is None else w
    _check(lib().moe_route_topk_static(_ptr(x), M, H, _ptr(Wr), E, _ptr(skew), k, _ptr(idx), _ptr(w),
                                       _stream(stream)), "moe_route_topk_static")
    return idx, w


def moe_expert_forward_decode(pool: Pool, x: torch.Tensor, idx: torch.Tensor, w: torch.Tensor,
                              residual: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                              y: torch.Tensor | None = None, stream=None):
    _need(x, torch.bfloat16, "x")
    _need(idx, torch.int32, "idx")
    _need(w, torch.float32, "w")
    M, k = idx.shape
    if residual is not None:
        _need(residual, torch.bfloat16, "residual")
    if ws is None:
        ws = workspace(moe_workspace_size(MOE_OP_DECODE, pool.E, pool.H, pool.I, M, k), x.device)
    y = torch.empty((M, pool.H), dtype=torch.bfloat16, device=x.device) if y is None else y
    _check(lib().moe_expert_forward_decode(pool.handle, _ptr(x), M, _ptr(idx), _ptr(w), k, _ptr(residual),
                                           _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_expert_forward_decode")
    return y


def moe_prescale(x: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    _need(x, torch.bfloat16, "x")
    M, H = x.shape
    out = torch.empty_like(x) if out is None else out
    _check(lib().moe_prescale(_ptr(x), M, H, _ptr(out), _stream(stream)), "moe_prescale")
    return out


def moe_expert_forward_grouped(pool: Pool, x: torch.Tensor, idx: torch.Tensor, act_mode: int = MOE_ACT_MXFP8,
                               partial_dtype: int = MOE_PARTIAL_F32, ws: torch.Tensor | None = None,
                               out: dict | None = None, stream=None):
    _need(x, torch.bfloat16, "x")
    _need(idx, torch.int32, "idx")
    T, k = idx.shape
    dev = x.device
    if ws is None:
        ws = workspace(moe_workspace_size(MOE_OP_GROUPED, pool.E, pool.H, pool.I, T, k), dev)
    if out is None:
        pdt = torch.float32 if partial_dtype == MOE_PARTIAL_F32 else torch.bfloat16
        out = {"perm": torch.empty(T * k, dtype=torch.int32, device=dev),
               "inv_perm": torch.empty(T * k, dtype=torch.int32, device=dev),
               "offsets": torch.empty(pool.E + 1, dtype=torch.int32, device=dev),
               "partial": torch.empty((T * k, pool.H), dtype=pdt, device=dev)}
    _check(lib().moe_expert_forward_grouped(pool.handle, _ptr(x), T, _ptr(idx), k, act_mode, _ptr(out["perm"]),
                                            _ptr(out["inv_perm"]), _ptr(out["offsets"]), _ptr(out["partial"]),
                                            partial_dtype, _ptr(ws), ws.numel(), _stream(stream)),
           "moe_expert_forward_grouped")
    return out


def moe_grouped_read_h(pool: Pool, T: int, k: int, offsets: torch.Tensor, ws: torch.Tensor,
                       act_mode: int = MOE_ACT_MXFP8, stream=None):
    """The MX-quantised h of the last grouped call on `ws`, in sorted row order:
    (codes uint8 [T*k, I] (E4M3, or E2M1 with MOE_ACT_MXFP4), scale bytes [T*k, I/32])."""
    _need(offsets, torch.int32, "offsets")
    hq = torch.zeros((T * k, pool.I), dtype=torch.uint8, device=ws.device)
    hs = torch.zeros((T * k, pool.I // 32), dtype=torch.uint8, device=ws.device)
    _check(lib().moe_grouped_read_h(pool.handle, T, k, act_mode, _ptr(offsets), _ptr(ws), ws.numel(), _ptr(hq),
                                    _ptr(hs), _stream(stream)), "moe_grouped_read_h")
    return hq, hs


def moe_combine(partial: torch.Tensor, inv_perm: torch.Tensor, w: torch.Tensor, residual: torch.Tensor | None = None,
                y: torch.Tensor | None = None, stream=None):
    _need(inv_perm, torch.int32, "inv_perm")
    _need(w, torch.float32, "w")
    T, k = w.shape
    H = partial.shape[1]
    pdt = MOE_PARTIAL_F32 if partial.dtype == torch.float32 else MOE_PARTIAL_BF16
    y = torch.empty((T, H), dtype=torch.bfloat16, device=partial.device) if y is None else y
    _check(lib().moe_combine(_ptr(partial), pdt, _ptr(inv_perm), _ptr(w), T, k, H, _ptr(residual), _ptr(y),
                             _stream(stream)), "moe_combine")
    return y


# ------------------------------------------------------ streamed expert pool


class _CacheView:
    """The device cache of a StreamPool, usable wherever a Pool is (slot indices)."""

    def __init__(self, handle, E, H, I, mem):
        self.handle, self.E, self.H, self.I, self.mem = handle, E, H, I, mem


class StreamPool:
    """Expert records in pinned host memory (`host`, a CPU uint8 tensor holding E
    records), an HBM cache of `slots` records; `cache` is the pool view the kernels use
    with the slot indices that `map` returns."""

    def __init__(self, host: torch.Tensor, E: int, H: int, I: int, slots: int, device="cuda", plan_only=False):
        if host.is_cuda or host.dtype != torch.uint8 or not host.is_contiguous():
            raise ValueError("host: expected a contiguous CPU uint8 tensor")
        self.E, self.H, self.I = E, H, I
        rec = moe_pool_record_bytes(H, I)
        self.host = host
        self.rec = rec
        if plan_only:
            self.buffer, mem, cache_ptr = None, None, None
        else:
            self.buffer = torch.empty(slots * rec + 1024, dtype=torch.uint8, device=device)
            off = (-self.buffer.data_ptr()) % 1024
            mem = self.buffer[off:off + slots * rec]
            cache_ptr = _ptr(mem)
        h = ctypes.c_void_p()
        _check(lib().moe_stream_pool_create(ctypes.byref(h), ctypes.c_void_p(host.data_ptr()), host.numel(), E, H, I,
                                            cache_ptr, slots * rec), "moe_stream_pool_create")
        self.handle = h
        self.slots = int(lib().moe_stream_pool_slots(h))
        c = lib().moe_stream_pool_cache(h)
        self.cache = None if c is None else _CacheView(ctypes.c_void_p(c), self.slots, H, I, mem)
        self._idx = torch.empty(32 * 32, dtype=torch.int32).pin_memory() if not plan_only else None

    def map(self, idx_host, stream=None):
        """Slots (int32 numpy array, same shape) for the expert indices `idx_host`
        (numpy int32); misses are copied on `stream` (the current stream if None)."""
        import numpy as np
        a = np.ascontiguousarray(idx_host, dtype=np.int32)
        out = np.empty_like(a)
        st = None if self.cache is None else _stream(stream)
        _check(lib().moe_stream_pool_map(self.handle, a.ctypes.data_as(ctypes.c_void_p), a.size,
                                         out.ctypes.data_as(ctypes.c_void_p), st), "moe_stream_pool_map")
        return out

    def stats(self):
        """(hits, misses, bytes copied) since creation."""
        h, m, b = _u64(), _u64(), _u64()
        _check(lib().moe_stream_pool_stats(self.handle, ctypes.byref(h), ctypes.byref(m), ctypes.byref(b)),
               "moe_stream_pool_stats")
        return int(h.value), int(m.value), int(b.value)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.moe_stream_pool_destroy(h)
            self.handle = None


class HostBuffer:
    """`nbytes` of pinned host memory on the NUMA node closest to `device`
    (moe_host_alloc); `tensor` is a CPU uint8 view of it, `numa_node` the node its
    first page lies on (-1 if unknown).  Freed by close() or when collected; the
    tensor must not be used after that."""

    def __init__(self, nbytes: int, device=None):
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.nbytes = int(nbytes)
        p, node = _vp(), _i()
        _check(lib().moe_host_alloc(dev.index or 0, self.nbytes, ctypes.byref(p), ctypes.byref(node)),
               "moe_host_alloc")
        self._p = p
        self.numa_node = int(node.value)
        arr = (ctypes.c_uint8 * self.nbytes).from_address(p.value)
        self.tensor = torch.frombuffer(arr, dtype=torch.uint8)

    def close(self):
        if getattr(self, "_p", None) is not None and _lib is not None:
            self.tensor = None
            _check(_lib.moe_host_free(self._p, self.nbytes), "moe_host_free")
            self._p = None

    def __del__(self):
        try:
            self.close()
        except MoeError:
            pass


def moe_host_numa_node(device=None) -> int:
    """The host NUMA node closest to `device` (-1: no NUMA or unknown)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    return int(lib().moe_host_numa_node(dev.index or 0))


CTA_PAIRS_NEVER, CTA_PAIRS_ALWAYS, CTA_PAIRS_MXFP8 = 0, 1, 2


def moe_grouped_set_cta_pairs(mode: int):
    """Tile shape of the grouped GEMMs for later calls: one-part tiles of 128+ columns on
    pairs of SMs (tcgen05 cta_group::2) never (0), always (1), or with MXFP8 rows only
    (2, the default)."""
    _check(lib().moe_grouped_set_cta_pairs(int(mode)), "moe_grouped_set_cta_pairs")


# ---------------------------------------------------------- test support


def moe_debug_set_wait_limit(ns: int):
    """Bound every device wait of the library by `ns` nanoseconds (0: the 1 s default)."""
    _check(lib().moe_debug_set_wait_limit(ns), "moe_debug_set_wait_limit")


def moe_debug_set_barrier_extra(extra: int):
    """Make the single-token decode kernel's grid barrier wait for `extra` arrivals
    that never come (0 turns the hook off)."""
    _check(lib().moe_debug_set_barrier_extra(extra), "moe_debug_set_barrier_extra")


# --------------------------------------------------------------- tracing


def moe_trace_begin(kernel_name: str):
    _check(lib().moe_trace_begin(kernel_name.encode()), "moe_trace_begin")


def moe_trace_end():
    """(launches, total device milliseconds) of the traced kernel since moe_trace_begin."""
    n = ctypes.c_int()
    ms = ctypes.c_double()
    _check(lib().moe_trace_end(ctypes.byref(n), ctypes.byref(ms)), "moe_trace_end")
    return int(n.value), float(ms.value)
