"""Helpers for the GPU parity tests: move generator output to the device."""
import numpy as np
import torch

DEV = torch.device("cuda:0")


def bf16_dev(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(DEV)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    diff = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return diff / den if den > 0 else diff


# tolerance for bf16 inputs and outputs with fp32 accumulation: max|err| <= 2e-2 * max|ref|
TOL = 2e-2
