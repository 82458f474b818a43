"""Shared helpers of the GPU parity tests (tensor marshalling and the tolerance)."""
import numpy as np
import torch

# Float tolerance of the layer output (stated with the routed-expert workload):
# max |err| <= 2e-2 * RMS(oracle) and relative L1 error <= 5e-3.
MAX_ERR_RMS = 2e-2
REL_L1 = 5e-3


def to_dev_bf16(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def check_close(y: np.ndarray, ref: np.ndarray, what: str = "y", amb=None):
    """The float tolerance; `amb` (optional, per element) adds the change that
    legitimate alternative MXFP8 roundings of h can explain (tensor-core path)."""
    err = np.abs(y - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    rel = float(err.sum() / max(np.abs(ref).sum(), 1e-300))
    if amb is not None:
        over = err - amb
        assert over.max() <= MAX_ERR_RMS * rms, (
            f"{what}: max(|err| - ambiguity) {over.max():.3e} > {MAX_ERR_RMS} * rms {rms:.3e}")
        assert rel <= REL_L1, f"{what}: relative L1 {rel:.3e} > {REL_L1}"
        return float(err.max() / rms), rel
    assert err.max() <= MAX_ERR_RMS * rms, f"{what}: max|err| {err.max():.3e} > {MAX_ERR_RMS} * rms {rms:.3e}"
    assert rel <= REL_L1, f"{what}: relative L1 {rel:.3e} > {REL_L1}"
    return float(err.max() / rms), rel
