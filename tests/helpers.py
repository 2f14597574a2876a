"""Shared test helpers: tolerance rule, tensor <-> numpy conversion."""
import numpy as np
import torch

import oracle

# Output tolerance (bf16 outputs, fp32 accumulation): rel-L2 against the oracle's
# bf16-rounded result <= 1e-3, and max |gpu - exact| <= 2e-2 * RMS(exact).
REL_L2 = 1e-3
MAX_ABS_RMS = 2e-2


def u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def bf16_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def assert_close_to_oracle(gpu: torch.Tensor, exact: np.ndarray, what: str = ""):
    g = bf16_f64(gpu).reshape(exact.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    rounded = oracle.bf16_bits_to_f64(oracle.bf16_round_array(exact))
    denom = np.linalg.norm(exact)
    rel = np.linalg.norm(g - rounded) / max(denom, 1e-300)
    rms = np.sqrt(np.mean(exact ** 2))
    mx = np.max(np.abs(g - exact))
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_RMS * rms + 1e-30, f"{what}: max-abs {mx:.3e} > {MAX_ABS_RMS} * rms {rms:.3e}"
    return rel, mx / max(rms, 1e-300)
