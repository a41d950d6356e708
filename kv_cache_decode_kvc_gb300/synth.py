"""Seeded synthetic inputs for the decode step (no attention arithmetic in here).

The same values must come out on the CPU (for the oracle) and on the GPU (for the
CUDA path), slice by slice, so the generator is counter-based: every element is a
pure function of (seed, layer, tensor, b, head, t, d).  It is written with torch
integer ops that give identical results on any device:

* a 32-bit hash of the element's 64-bit counter and a second 32-bit value hashed from the
  first (the murmur3 finaliser, with every product split into 16-bit halves so no int64 ever
  overflows);
* their four 16-bit halves u_1..u_4 are summed: an Irwin-Hall(4) draw on a grid of 2^-16,
  centred and scaled by one IEEE fp32 multiplication to mean 0 and standard deviation 1
  (support [-3.46, 3.46]), then rounded to the requested dtype (bf16: nearest even).  The
  bell-shaped unit-variance draw stands in for N(0, 1); the fine grid makes the bf16 values
  use their whole significand, so products and sums round as they do on real activations.

Lengths and the small worked example use torch's CPU generator (seeded), which is
device-independent because they are drawn on the host.
"""
from __future__ import annotations

import torch

TENSOR_IDS = {"K": 0, "V": 1, "Q": 2}
T_STRIDE = 1 << 21          # counter slots per (b, head) stream: covers T up to 2M
_M32 = 0xFFFFFFFF


def _mul32(h: torch.Tensor, c: int) -> torch.Tensor:
    """(h * c) mod 2^32 for int64 tensors holding values in [0, 2^32), without overflow."""
    lo = h & 0xFFFF
    hi = h >> 16
    return ((lo * c) + (((hi * c) & 0xFFFF) << 16)) & _M32


def _fmix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    return h ^ (h >> 16)


_SALT_A = 0x9E3779B9
_SALT_B = 0x7F4A7C15
# 1 / sqrt(var(u_1 + u_2 + u_3 + u_4)) for u_i uniform on {0 .. 65535}: var = (65536^2 - 1) / 3
_UNIT = float(torch.tensor(1.0 / ((65536.0 ** 2 - 1.0) / 3.0) ** 0.5, dtype=torch.float32))


def _fmix32_int(h: int) -> int:
    """_fmix32 of one Python integer (the seed's part of the hash, computed once)."""
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & _M32
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & _M32
    return h ^ (h >> 16)


def _hash(lo: torch.Tensor, hi: torch.Tensor, seed: int, salt: int) -> torch.Tensor:
    s = _fmix32_int((seed ^ salt) & _M32)
    return _fmix32(lo ^ _fmix32(hi ^ s))


def hash_values(counter: torch.Tensor, seed: int) -> torch.Tensor:
    """float32 values (see module doc) for int64 counters >= 0."""
    lo = counter & _M32
    hi = counter >> 32
    a = _hash(lo, hi, seed, _SALT_A)
    b = _fmix32(a ^ _SALT_B)  # a second 32-bit draw from the first
    total = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16)
    # |total - 131070| < 2^24: exact in fp32; one rounded multiplication on any device
    unit = torch.tensor(_UNIT, dtype=torch.float32, device=counter.device)
    return (total - 131070).to(torch.float32) * unit


def rows(seed: int, layer: int, tensor: str, b: int, head: int, t0: int, t1: int, D: int,
         n_batch: int, n_heads: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """Rows t0..t1-1 of one (b, head) stream of one tensor: shape [t1-t0, D]."""
    base = ((((layer * 4 + TENSOR_IDS[tensor]) * n_batch + b) * n_heads + head) * T_STRIDE)
    t = torch.arange(t0, t1, device=device, dtype=torch.int64).unsqueeze(1)
    d = torch.arange(D, device=device, dtype=torch.int64).unsqueeze(0)
    ctr = (base + t) * D + d
    return hash_values(ctr, seed).to(dtype)


def block(seed: int, layer: int, tensor: str, b0: int, b1: int, n_heads: int, t0: int, t1: int,
          D: int, n_batch: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """Rows t0..t1-1 of every head of batches b0..b1-1: shape [b1-b0, n_heads, t1-t0, D]."""
    tid = TENSOR_IDS[tensor]
    b = torch.arange(b0, b1, device=device, dtype=torch.int64).view(-1, 1, 1, 1)
    h = torch.arange(n_heads, device=device, dtype=torch.int64).view(1, -1, 1, 1)
    t = torch.arange(t0, t1, device=device, dtype=torch.int64).view(1, 1, -1, 1)
    d = torch.arange(D, device=device, dtype=torch.int64).view(1, 1, 1, -1)
    base = (((layer * 4 + tid) * n_batch + b) * n_heads + h) * T_STRIDE
    ctr = (base + t) * D + d
    return hash_values(ctr, seed).to(dtype)


def queries(seed: int, layer: int, B: int, H_q: int, D: int, dtype=torch.bfloat16,
            device="cpu") -> torch.Tensor:
    """q [B, H_q, D]: row 0 of each (b, query head) stream of tensor 'Q'."""
    return block(seed, layer, "Q", 0, B, H_q, 0, 1, D, B, dtype, device).squeeze(2).contiguous()


def uniform_lens(seed: int, B: int, lo: int, hi: int) -> torch.Tensor:
    """Cached lengths T_b ~ U{lo..hi} (inclusive), int32, drawn on the CPU generator."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def worked_example(seed: int = 7, hidden: int = 16, H_q: int = 4, H_kv: int = 2, D: int = 4,
                   B: int = 1, T: int = 13):
    """The glossary page's worked example inputs, drawn in its order on a CPU generator:
    W_Q [hidden, H_q*D], W_K [hidden, H_kv*D], W_V [hidden, H_kv*D], W_O [H_q*D, hidden],
    each randn / sqrt(hidden), then x = randn [B, T, hidden]; fp32."""
    g = torch.Generator().manual_seed(seed)
    shapes = [(hidden, H_q * D), (hidden, H_kv * D), (hidden, H_kv * D), (H_q * D, hidden)]
    Ws = [torch.randn(s, generator=g, dtype=torch.float32) / hidden ** 0.5 for s in shapes]
    x = torch.randn(B, T, hidden, generator=g, dtype=torch.float32)
    return Ws, x


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 CPU tensor (the oracle's bf16 input format)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
