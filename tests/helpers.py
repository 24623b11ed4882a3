"""Shared test helpers: bit views of bf16 / fp16 / fp32 tensors and ulp distances."""
import numpy as np
import torch


def bits(t):
    """bf16 torch tensor (any device) -> uint16 numpy bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(b, device="cpu"):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_ulp_distance(a_bits, b_bits):
    """Distance in bf16 units in the last place (+0 and -0 are the same point)."""
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def ulp_distance(a_bits, b_bits):
    """Distance in units in the last place between two arrays of IEEE bit patterns of
    the same width (uint16 for bf16 / fp16, uint32 for fp32); +0 and -0 coincide."""
    a_bits = np.asarray(a_bits)
    b_bits = np.asarray(b_bits)
    width = a_bits.dtype.itemsize * 8
    sign = 1 << (width - 1)

    def ordered(u):
        u = u.astype(np.int64)
        return np.where(u & sign, -(u & (sign - 1)), u)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def out_bits(t):
    """bf16 / fp16 / fp32 torch tensor -> numpy IEEE bit patterns (uint16 or uint32)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


# The floating-point tolerance of the fused epilogue: at most 1 bf16 ulp from the
# oracle (the same fp32 operation order gives 0; the bound admits a different but
# still correctly-rounded-per-step evaluation).
MAX_ULP = 1
