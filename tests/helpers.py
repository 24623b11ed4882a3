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


# The tolerance of the INT8 path's outputs against the oracle, in ulps of the output
# type: 0.  The kernel evaluates the epilogue in the oracle's fp32 operation order, each
# step rounded on its own, from the same exact int32 accumulator and the same scales, so
# every output bit must agree (the 16-bit-activation path has its own derived bound).
MAX_ULP = 0


# ---- guard bands: outputs placed inside a larger buffer whose every element starts as a
# bit pattern the computation never produces.  After the call, every element of the
# output must have been overwritten (no skipped or mis-addressed tile) and the bands on
# both sides must be untouched (no write past either end).
GUARD = 2048  # elements on each side (a multiple of 256 bytes for every element size)
_INT_OF = {1: torch.int8, 2: torch.int16, 4: torch.int32}


def _signed(pattern, nbytes):
    bits_ = 8 * nbytes
    pattern &= (1 << bits_) - 1
    return pattern - (1 << bits_) if pattern >> (bits_ - 1) else pattern


def guarded(shape, dtype, pattern, device="cuda"):
    """(buffer, view): `view` of `shape` and `dtype` inside `buffer`, all of it filled with
    the raw bit pattern `pattern` (e.g. 0x7FFF, a bf16 / fp16 NaN; -128 for int8 codes,
    which the clamp to [-127, 127] never writes)."""
    n = 1
    for d in shape:
        n *= int(d)
    size = torch.empty((), dtype=dtype).element_size()
    buf = torch.full((n + 2 * GUARD,), _signed(pattern, size), dtype=_INT_OF[size], device=device)
    view = buf[GUARD:GUARD + n].view(dtype).view(*shape)
    return buf, view


def assert_guards_intact(buf, pattern):
    size = buf.element_size()
    p = _signed(pattern, size)
    assert bool((buf[:GUARD] == p).all()), "a write landed in the guard band before the output"
    assert bool((buf[-GUARD:] == p).all()), "a write landed in the guard band after the output"


def assert_all_written(buf, pattern, chunk=1 << 28):
    """No element between the guard bands still holds the fill pattern (checked on the
    device, in chunks)."""
    p = _signed(pattern, buf.element_size())
    body = buf[GUARD:buf.numel() - GUARD]
    for i in range(0, body.numel(), chunk):
        left = int((body[i:i + chunk] == p).sum())
        assert left == 0, "%d output elements were never written (first chunk at %d)" % (left, i)


NAN16 = 0x7FFF        # bf16 and fp16 NaN
NAN32 = 0x7FFFFFFF    # fp32 NaN
CODE_NEVER = -128     # int8 code the symmetric clamp never produces
ACC_NEVER = -(1 << 31)  # int32 accumulator below -127*127*131072


def guarded_workspace(nbytes, device="cuda", seed=0):
    """A workspace of nbytes random bytes between two guard bands of random bytes;
    returns (buffer, workspace view, copy of the buffer) -- compare the bands after."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    buf = torch.randint(0, 256, (nbytes + 2 * GUARD * 16,), dtype=torch.uint8, device=device, generator=g)
    return buf, buf[GUARD * 16:GUARD * 16 + nbytes], buf.clone()


def assert_workspace_guards_intact(buf, before):
    G = GUARD * 16
    assert torch.equal(buf[:G], before[:G]), "a write landed before the workspace"
    assert torch.equal(buf[-G:], before[-G:]), "a write landed after the workspace"
