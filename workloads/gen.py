"""Seeded, device-independent synthetic values.

Both sides of every parity check draw their inputs from here: the CUDA path
generates whole workloads on the GPU, the CPU oracle regenerates the rows it
needs on the host, and the two get bit-identical values.  That works because
every step is integer arithmetic or an exactly rounded fp32 operation:

* ``mix32`` -- a two-round xor-shift/multiply 32-bit hash.  Both multipliers
  are below 2^31, so every product of a 32-bit value fits in int64 without
  overflow; results are masked back to 32 bits.
* ``normal`` -- a discretised N(0, 1): the hash's top 16 bits select one of
  65536 equiprobable standard-normal quantiles, Phi^-1((i + 1/2) / 65536),
  tabulated once on the host in fp64 and rounded to fp32 (support about
  [-4.3, 4.3]).  The same table is copied to every device, so a value depends
  only on (key, index).

Nothing here knows about attention, caches or slots: it only maps
(seed, role, sequence, element index) to a number.
"""
from __future__ import annotations

import torch

M32 = 0xFFFFFFFF
_C1 = 0x21F0AAAD
_C2 = 0x735A2D97
_GOLD = 0x9E3779B9

# roles keep the streams of different tensors apart
ROLE = {"q": 1, "k_hist": 2, "v_hist": 3, "k_step": 4, "v_step": 5, "outlier": 6, "pad": 7}

_CHUNK = 1 << 24  # elements per generation chunk (bounds temporary memory)


def mix32(x: torch.Tensor) -> torch.Tensor:
    """32-bit hash of int64 values in [0, 2^32)."""
    x = x ^ (x >> 16)
    x = (x * _C1) & M32
    x = x ^ (x >> 15)
    x = (x * _C2) & M32
    x = x ^ (x >> 15)
    return x


def _mix_int(v: int) -> int:
    v &= M32
    v ^= v >> 16
    v = (v * _C1) & M32
    v ^= v >> 15
    v = (v * _C2) & M32
    v ^= v >> 15
    return v


def stream_key(seed: int, role: str, seq: int) -> int:
    """32-bit key of the stream (seed, role, sequence)."""
    k = _mix_int(seed ^ _mix_int(seed >> 32))
    k = _mix_int(k ^ (ROLE[role] * _GOLD & M32))
    k = _mix_int(k ^ (seq * 0x85EBCA6B & M32) ^ 0x5BD1E995)
    return k


_TABLE_CPU = None
_TABLES = {}


def quantile_table(device="cpu") -> torch.Tensor:
    """fp32 [65536]: Phi^-1((i + 1/2) / 65536), computed on the host, copied as is."""
    global _TABLE_CPU
    if _TABLE_CPU is None:
        u = (torch.arange(65536, dtype=torch.float64) + 0.5) / 65536.0
        _TABLE_CPU = torch.special.ndtri(u).to(torch.float32)
    key = str(torch.device(device))
    if key not in _TABLES:
        _TABLES[key] = _TABLE_CPU.to(device)
    return _TABLES[key]


def normal_from_keys(keys: torch.Tensor, idx: torch.Tensor) -> torch.Tensor:
    """Approximately N(0,1) fp32 values for int64 (key, index) pairs (same shape)."""
    h = mix32((idx & M32) ^ keys)
    h = mix32(h ^ (keys >> 7))
    return quantile_table(idx.device)[h >> 16]


def normal(seed: int, role: str, seq: int, n: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """n values of stream (seed, role, seq), element indices offset .. offset+n-1."""
    key = stream_key(seed, role, seq)
    out = torch.empty(n, dtype=torch.float32, device=device)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        idx = torch.arange(offset + c0, offset + c1, dtype=torch.int64, device=device)
        keys = torch.full_like(idx, key)
        out[c0:c1] = normal_from_keys(keys, idx)
    return out


def rows(seed: int, role: str, seqs, positions, width: int, device="cpu", cols=None) -> torch.Tensor:
    """Rows of a stream laid out `width` values per position: row r holds elements
    [pos*width, (pos+1)*width) of stream (seed, role, seqs[r]), or only the columns
    `cols` of it.  seqs/positions: 1-D int sequences of equal length.
    Returns fp32 [R, width] (or [R, len(cols)])."""
    seqs = torch.as_tensor(seqs, dtype=torch.int64)
    positions = torch.as_tensor(positions, dtype=torch.int64)
    R = int(seqs.numel())
    col = torch.arange(width, dtype=torch.int64) if cols is None else torch.as_tensor(cols, dtype=torch.int64)
    C = int(col.numel())
    col = col.to(device)
    out = torch.empty((R, C), dtype=torch.float32, device=device)
    if R == 0:
        return out
    uniq = torch.unique(seqs).tolist()
    keymap = {s: stream_key(seed, role, s) for s in uniq}
    row_keys = torch.tensor([keymap[int(s)] for s in seqs.tolist()], dtype=torch.int64)
    rows_per_chunk = max(1, _CHUNK // C)
    for r0 in range(0, R, rows_per_chunk):
        r1 = min(R, r0 + rows_per_chunk)
        k = row_keys[r0:r1].to(device)[:, None].expand(r1 - r0, C)
        idx = positions[r0:r1].to(device)[:, None] * width + col[None, :]
        out[r0:r1] = normal_from_keys(k, idx)
    return out
