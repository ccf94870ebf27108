"""Raw-bit conversions for test inputs, done with numpy/torch (not the oracle).

Input plumbing: the values handed in are exactly representable in the target
type wherever a test relies on that, so the conversion does not round.
"""
import numpy as np
import torch

TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}
BITS = {"f32": (torch.int32, np.uint32), "f16": (torch.int16, np.uint16),
        "bf16": (torch.int16, np.uint16), "e4m3": (torch.uint8, np.uint8)}
NBYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}


def to_bits(values, dtype):
    """float64 array -> raw bit array of `dtype` (rounding through torch)."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float64))
    if dtype in ("bf16", "e4m3"):
        t = t.to(torch.float32)
    t = t.to(TORCH[dtype])
    ti, npi = BITS[dtype]
    return t.view(ti).numpy().view(npi).copy()


def from_bits(bits, dtype):
    """raw bit array -> float64 values (through torch)."""
    return torch_from_bits(bits, dtype).to(torch.float64).numpy()


def torch_from_bits(bits, dtype):
    ti, npi = BITS[dtype]
    signed = {np.uint32: np.int32, np.uint16: np.int16, np.uint8: np.uint8}[npi]
    arr = np.ascontiguousarray(np.asarray(bits).astype(npi))
    return torch.from_numpy(arr.view(signed)).view(TORCH[dtype])


def bits_of_tensor(t):
    name = {v: k for k, v in TORCH.items()}[t.dtype]
    ti, npi = BITS[name]
    return t.contiguous().view(ti).cpu().numpy().view(npi)
