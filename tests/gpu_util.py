"""Helpers for GPU tests: move seeded numpy inputs to the device and back."""
from __future__ import annotations

import numpy as np
import torch

import lrkv_synth as S


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> device bfloat16 tensor (same bits)."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Device bfloat16 tensor -> uint16 numpy bits."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return S.bf16_bits_to_f32(host_bits(t)).astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(got - ref))) if got.size else 0.0
    return rel, mx


# Parity bar for decode and prefill outputs (relative L2 and max abs against the fp64 oracle).
REL_L2_TOL = 5e-3
MAX_ABS_TOL = 2e-2


def assert_close(got, ref, what=""):
    rel, mx = errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, f"{what}: rel_l2={rel:.3e} max_abs={mx:.3e}"
    return rel, mx
