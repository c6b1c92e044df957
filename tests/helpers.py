"""Test-side conversions between torch tensors and the oracle's storage form."""
import numpy as np
import torch


def to_store(t: torch.Tensor) -> np.ndarray:
    """Raw element storage: float32 stays float32, bfloat16 becomes uint16 bits,
    e4m3 code caches (uint8) stay uint8."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.float32, torch.uint8):
        return t.numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(t.dtype)


def dtype_name(t: torch.Tensor) -> str:
    return {torch.float32: "f32", torch.bfloat16: "bf16"}[t.dtype]


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values through torch's own conversion (independent of the oracle)."""
    return t.detach().cpu().to(torch.float64).numpy()
