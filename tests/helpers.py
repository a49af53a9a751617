"""Test-side helpers: tensor conversion, layout decoding and error metrics.

These hold no arithmetic of the layer itself; they move data between torch,
numpy and the documented device layouts.
"""
import numpy as np
import torch


def f64(t):
    """torch tensor (any float dtype, any device) -> float64 numpy."""
    return t.detach().to("cpu", torch.float64).numpy()


def u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def i32(t):
    return t.detach().cpu().numpy().astype(np.int64)


def scales_tiled_to_rowmajor(s, mn, kdim):
    """Decode the 512-byte tiled scale layout of include/moe.h to [mn, kdim/32]."""
    s = np.asarray(s, dtype=np.uint8).reshape(mn // 128, kdim // 128, 32, 4, 4)
    return s.transpose(0, 3, 2, 1, 4).reshape(mn, kdim // 32)


def scales_rowmajor_to_tiled(s, mn, kdim):
    """Inverse of scales_tiled_to_rowmajor: [mn, kdim/32] to the tiled bytes."""
    s = np.asarray(s, dtype=np.uint8).reshape(mn // 128, 4, 32, kdim // 128, 4)
    return np.ascontiguousarray(s.transpose(0, 3, 2, 1, 4)).reshape(-1)


def rel_fro(a, ref):
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))


def max_abs_rel(a, ref):
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    m = np.max(np.abs(ref)) if ref.size else 0.0
    return float(np.max(np.abs(a - ref)) / (m if m > 0 else 1.0)) if ref.size else 0.0


def bf16_round(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64)).to(torch.float32).to(
        torch.bfloat16).to(torch.float64).numpy()
