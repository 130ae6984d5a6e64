"""Materialise a workload's values on any device (bit-identical everywhere).

* ``q(w)``              [S * nq, Hq, D] (nq query tokens per sequence)
* ``history_rows(w, s)`` K, V rows of positions [0, L_s) of sequence s, as the
                        history written before the measured step
* ``step_rows(w)``      K, V rows of the measured step [T, Hkv, D]
* ``logical_kv(w, s)``  the sequence's K, V in logical order after the step:
                        history, with the positions the step writes (slot >= 0)
                        replaced by the step rows

Values are rounded to the workload dtype (RNE); fp8 quantisation is not done
here -- each side does its own.
"""
from __future__ import annotations

import torch

from . import gen
from .configs import Workload

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _round(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(TORCH_DT[dtype])


def q(w: Workload, device="cpu") -> torch.Tensor:
    """[S * nq, Hq, D]: query token i of sequence s is row s * nq + i (position index i of the
    sequence's q stream)."""
    seqs = [s for s in range(w.S) for _ in range(w.nq)]
    pos = [i for _ in range(w.S) for i in range(w.nq)]
    vals = gen.rows(w.seed, "q", seqs, pos, w.Hq * w.D, device=device)
    return _round(vals.view(w.S * w.nq, w.Hq, w.D), w.dtype)


def _outlier_rows(w: Workload, s: int) -> torch.Tensor:
    """K row at the outlier position of sequence s: for each KV head g,
    (target / (scale * |q_h0|^2)) * q_h0 with h0 = g * G, so that head h0's logit is
    about `target`.  Computed on the CPU in fp32 and rounded to the workload dtype."""
    target = float(w.notes.get("outlier_logit", 20.0))
    qs = q(w, "cpu")[s].float()                      # [Hq, D]
    rows = torch.empty((w.Hkv, w.D), dtype=torch.float32)
    for g in range(w.Hkv):
        q0 = qs[g * w.G]
        rows[g] = q0 * (target / (w.scale * float((q0 * q0).sum())))
    return _round(rows, w.dtype)


def _cols(w: Workload, kv_heads):
    if kv_heads is None:
        return None, w.Hkv
    kv_heads = list(kv_heads)
    cols = torch.cat([torch.arange(g * w.D, (g + 1) * w.D) for g in kv_heads])
    return cols, len(kv_heads)


def history_rows(w: Workload, s: int, device="cpu", positions=None, kv_heads=None):
    """(K, V) history rows of sequence s at `positions` (default all of [0, L_s)),
    optionally only for the KV heads `kv_heads` ([n, len(kv_heads), D])."""
    L = int(w.seq_lens[s])
    if positions is None:
        positions = torch.arange(L, dtype=torch.int64)
    positions = torch.as_tensor(positions, dtype=torch.int64)
    n = int(positions.numel())
    seqs = torch.full((n,), s, dtype=torch.int64)
    width = w.Hkv * w.D
    cols, nh = _cols(w, kv_heads)
    K = _round(gen.rows(w.seed, "k_hist", seqs, positions, width, device, cols), w.dtype).view(n, nh, w.D)
    V = _round(gen.rows(w.seed, "v_hist", seqs, positions, width, device, cols), w.dtype).view(n, nh, w.D)
    if w.outlier_pos is not None:
        hit = (positions == int(w.outlier_pos[s])).nonzero().flatten()
        if hit.numel():
            orow = _outlier_rows(w, s)
            if kv_heads is not None:
                orow = orow[list(kv_heads)]
            K[hit.to(K.device)] = orow.to(device)
    return K, V


def step_rows(w: Workload, device="cpu"):
    """(K, V) rows of the measured step, [T, Hkv, D]; rows with seq = -1 hold NaN."""
    seqs = torch.as_tensor(w.step_seq, dtype=torch.int64)
    pos = torch.as_tensor(w.step_pos, dtype=torch.int64)
    width = w.Hkv * w.D
    real = seqs >= 0
    sq = torch.where(real, seqs, torch.zeros_like(seqs))
    K = gen.rows(w.seed, "k_step", sq, pos, width, device).view(-1, w.Hkv, w.D)
    V = gen.rows(w.seed, "v_step", sq, pos, width, device).view(-1, w.Hkv, w.D)
    nan = (~real).to(device)
    K[nan] = float("nan")
    V[nan] = float("nan")
    return _round(K, w.dtype), _round(V, w.dtype)


def logical_kv(w: Workload, s: int, device="cpu", kv_heads=None):
    """Sequence s's K, V [L_s, Hkv, D] in logical order, after the step
    (optionally only the KV heads `kv_heads`)."""
    K, V = history_rows(w, s, device, kv_heads=kv_heads)
    sel = [(i, int(p)) for i, (sq, p, sl) in enumerate(zip(w.step_seq, w.step_pos, w.step_slot))
           if int(sq) == s and int(sl) >= 0]
    if sel:
        Ks, Vs = step_rows_subset(w, [i for i, _ in sel], device)
        if kv_heads is not None:
            Ks, Vs = Ks[:, list(kv_heads)], Vs[:, list(kv_heads)]
        idx = torch.tensor([p for _, p in sel], dtype=torch.int64, device=K.device)
        K[idx] = Ks
        V[idx] = Vs
    return K, V


def step_rows_subset(w: Workload, rows_idx, device="cpu"):
    """Step rows with the given row indices (all must belong to real sequences)."""
    seqs = torch.as_tensor(w.step_seq[rows_idx], dtype=torch.int64)
    pos = torch.as_tensor(w.step_pos[rows_idx], dtype=torch.int64)
    assert bool((seqs >= 0).all())
    width = w.Hkv * w.D
    K = gen.rows(w.seed, "k_step", seqs, pos, width, device).view(-1, w.Hkv, w.D)
    V = gen.rows(w.seed, "v_step", seqs, pos, width, device).view(-1, w.Hkv, w.D)
    return _round(K, w.dtype), _round(V, w.dtype)
