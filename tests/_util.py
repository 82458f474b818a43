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


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |v| (8 significant bits; subnormal spacing 2^-133):
    the largest error of rounding v to bf16."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(np.maximum(e, -126.0) - 8)


def check_close(y: np.ndarray, ref: np.ndarray, what: str = "y", amb=None, bf16_at=None, l1_on=None):
    """The float tolerance: max|y - ref| <= 2e-2 * RMS(ref), relative L1 <= 5e-3, with
    two per-element allowances that name a stated rounding step:
      - `amb` (tensor-core prefill path): the largest change that equally valid MXFP8
        roundings of h can make (the oracle's error model of the GPU's fp32 h); the
        elements that need it must be rare;
      - `bf16_at`: the values that were rounded to the stated bf16 output format (the
        GPU output itself, or the residual stream it was fused with); each element may
        also differ by the half-ulp of that rounding, which at |y| beyond about
        10 * RMS exceeds 2e-2 * RMS by itself.
    `l1_on` = (output, reference) on which the relative L1 error is taken when that
    is not (y, ref): for a layer fused with its residual, the max error is judged on
    the MoE part and the relative L1 on the layer's output, the residual stream."""
    err = np.abs(y - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    yl, rl = (y, ref) if l1_on is None else l1_on
    rel = float(np.abs(yl - rl).sum() / max(np.abs(rl).sum(), 1e-300))
    tol = MAX_ERR_RMS * rms
    allow = np.zeros_like(err) if bf16_at is None else bf16_half_ulp(np.abs(bf16_at) + tol)
    over = err - allow
    need, slack = 0.0, 0.0
    if amb is not None:
        assert (over - amb).max() <= tol, (
            f"{what}: max(|err| - allowances) {(over - amb).max():.3e} > {MAX_ERR_RMS} * rms {rms:.3e}")
        need = float(np.mean(over > tol))
        slack = float(np.max(amb) / rms) if rms > 0 else 0.0
        assert need <= SLACK_FRAC, f"{what}: {need:.2e} of the elements need the ambiguity slack"
    else:
        assert over.max() <= tol, f"{what}: max(|err| - bf16 allowance) {over.max():.3e} > {MAX_ERR_RMS} * rms {rms:.3e}"
    assert rel <= REL_L1, f"{what}: relative L1 {rel:.3e} > {REL_L1}"
    MARGINS.append({"what": what, "max_err_rms": float(err.max() / rms) if rms > 0 else 0.0, "rel_l1": rel,
                    "max_slack_rms": slack, "slack_frac": need,
                    "bf16_frac": float(np.mean(err > tol)) if bf16_at is not None else 0.0, "n": int(err.size)})
    return float(err.max() / rms) if rms > 0 else 0.0, rel


def report_close(y: np.ndarray, ref: np.ndarray, what: str, rel_l1: float = REL_L1):
    """Record max|err|/RMS and relative L1 of a comparison whose per-element bound does
    not apply as such (an end-to-end pass in which each side feeds its own rounded
    outputs forward), and assert a relative L1 bound only (`rel_l1`)."""
    err = np.abs(y - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    rel = float(err.sum() / max(np.abs(ref).sum(), 1e-300))
    MARGINS.append({"what": what, "max_err_rms": float(err.max() / rms) if rms > 0 else 0.0, "rel_l1": rel,
                    "max_slack_rms": 0.0, "slack_frac": 0.0, "bf16_frac": float(np.mean(err > MAX_ERR_RMS * rms)),
                    "n": int(err.size)})
    assert rel <= rel_l1, f"{what}: relative L1 {rel:.3e} > {rel_l1}"
    return float(err.max() / rms) if rms > 0 else 0.0, rel
