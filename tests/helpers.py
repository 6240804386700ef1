"""Shared test helpers: device transfer and the numeric parity checks."""
import numpy as np
import torch

REL_L2_TOL = 1e-3        # relative L2 error of the layer output vs the oracle
MAX_ABS_FRAC_TOL = 1e-2  # max abs error / max |oracle output|
PARITY_REPORT = []       # (case, rel L2, max abs / max|ref|) of every check, printed by conftest


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def to_dev_bf16(x_bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(dev).view(torch.bfloat16)


def from_dev_bf16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def planes_to_dev(planes: dict, dev="cuda") -> dict:
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in planes.items()}


def assert_close_layer(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, what: str = ""):
    """The layer-output bar: rel L2 <= 1e-3 and max abs <= 1e-2 * max|ref|."""
    g = bf16_to_f64(y_gpu_bits)
    r = bf16_to_f64(y_ref_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    denom = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / max(denom, 1e-300)
    mx = np.max(np.abs(g - r)) if g.size else 0.0
    lim = MAX_ABS_FRAC_TOL * (np.max(np.abs(r)) if r.size else 0.0)
    PARITY_REPORT.append((what, float(rel), float(mx / np.max(np.abs(r))) if lim > 0 else 0.0))
    assert rel <= REL_L2_TOL, f"{what}: rel L2 {rel:.3e} > {REL_L2_TOL}"
    assert mx <= lim, f"{what}: max abs {mx:.3e} > {lim:.3e}"
    return rel, mx
