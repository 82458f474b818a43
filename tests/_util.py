"""Shared helpers of the GPU parity tests (tensor marshalling and the tolerance)."""
import numpy as np
import torch

# Float tolerance of the layer output (stated with the routed-expert workload):
# max |err| <= 2e-2 * RMS(oracle) and relative L1 error <= 5e-3.
MAX_ERR_RMS = 2e-2
REL_L1 = 5e-3
# Elements whose error exceeds 2e-2 * RMS and is explained only by the MXFP8-h
# ambiguity (see check_close) must stay this rare.
SLACK_FRAC = 1e-3

# Every comparison made through check_close in this process: what was compared, its
# max|err|/RMS, relative L1 error, the largest ambiguity slack (as a fraction of RMS)
# and the share of elements that needed it.  Printed in the terminal summary.
MARGINS = []


def dequant_mxfp4(codes, scales, rows, K):
    """Dense matrix [rows][K] from logical MXFP4 bytes (two E2M1 codes per byte, element
    2j in the low nibble; one E8M0 scale byte per 32 along K), by the OCP bit-field
    definition, independently of the oracle."""
    c = np.asarray(codes, dtype=np.uint8).reshape(rows, K // 2)
    nib = np.empty((rows, K), dtype=np.int64)
    nib[:, 0::2] = c & 15
    nib[:, 1::2] = c >> 4
    s, e, m = nib >> 3, (nib >> 1) & 3, nib & 1
    mag = np.where(e == 0, m * 0.5, np.exp2(e - 1.0) * (1 + m / 2))
    val = np.where(s == 1, -mag, mag)
    sc = np.exp2(np.asarray(scales, dtype=np.float64).reshape(rows, K // 32) - 127)
    return val * np.repeat(sc, 32, axis=1)


def split_expert(codes, scales, H, I):
    """(gate, up, down) parts of an expert's logical codes and scale bytes."""
    n1, n2 = I * H // 2, 2 * I * H // 2
    s1, s2 = I * H // 32, 2 * I * H // 32
    return ((codes[:n1], scales[:s1]), (codes[n1:n2], scales[s1:s2]), (codes[n2:], scales[s2:]))


def to_dev_bf16(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def check_close(y: np.ndarray, ref: np.ndarray, what: str = "y", amb=None):
    """The float tolerance.  `amb` (optional, per element; tensor-core prefill path)
    is the largest change that equally valid MXFP8 roundings of h can make to each
    output (the oracle's error model of the GPU's fp32 h): an element may exceed
    2e-2 * RMS by at most its amb, and such elements must be rare."""
    err = np.abs(y - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    rel = float(err.sum() / max(np.abs(ref).sum(), 1e-300))
    tol = MAX_ERR_RMS * rms
    need, slack = 0.0, 0.0
    if amb is not None:
        over = err - amb
        assert over.max() <= tol, f"{what}: max(|err| - ambiguity) {over.max():.3e} > {MAX_ERR_RMS} * rms {rms:.3e}"
        need = float(np.mean(err > tol))
        slack = float(np.max(amb) / rms) if rms > 0 else 0.0
        assert need <= SLACK_FRAC, f"{what}: {need:.2e} of the elements need the ambiguity slack"
    else:
        assert err.max() <= tol, f"{what}: max|err| {err.max():.3e} > {MAX_ERR_RMS} * rms {rms:.3e}"
    assert rel <= REL_L1, f"{what}: relative L1 {rel:.3e} > {REL_L1}"
    MARGINS.append({"what": what, "max_err_rms": float(err.max() / rms) if rms > 0 else 0.0, "rel_l1": rel,
                    "max_slack_rms": slack, "slack_frac": need, "n": int(err.size)})
    return float(err.max() / rms) if rms > 0 else 0.0, rel
