"""bf16 <-> float helpers for tests (bit-level, numpy)."""
import numpy as np
import torch


def to_bits(x) -> np.ndarray:
    """float array -> bf16 bit patterns (round to nearest even), uint16."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_float(bits) -> np.ndarray:
    """bf16 bit patterns -> exact float32."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)
