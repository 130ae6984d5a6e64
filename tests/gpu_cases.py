"""Decode test cases built on the host, independently of the library's write kernel.

The logical K/V of every sequence is drawn on the CPU (seeded torch generator),
placed into a NaN-poisoned physical pool by plain tensor indexing through a
seeded block permutation, and copied to the GPU.  For E4M3 caches the codes
are produced by the oracle's own quantiser.  The expected output is the
oracle's dense fp64 attention over the logical K/V (it never sees the block
table)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

B = 16


def within_tol(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """|got - ref| <= 1e-3 + ulp_bf16(ref), ulp_bf16(v) = 2^(max(floor(log2|v|), -126) - 7)."""
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.abs(ref)))
    ulp = np.exp2(np.maximum(e, -126) - 7)
    return np.abs(got - ref) <= 1e-3 + ulp


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ok = within_tol(got, ref)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        err = np.abs(got - ref)
        raise AssertionError("%s: %d of %d outside 1e-3 + 1 bf16 ulp; max err %.3g; first %s (got %s ref %s)"
                             % (what, (~ok).sum(), ok.size, np.nanmax(err), idx.tolist(),
                                [got[tuple(i)] for i in idx], [ref[tuple(i)] for i in idx]))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class Case:
    pass


def make_case(S, Hq, Hkv, D, lens, dtype=torch.bfloat16, fp8=False, seed=0, k_scale=1.0, v_scale=1.0,
              extra_blocks=5, table_pad=-1, kv_sigma=1.0, perm=None, nhd=False, alibi=None) -> Case:
    """k_scale / v_scale: one FP8 scale, or Hkv per-head scales.  nhd: caches stored token-major
    within a block ([NB, 16, Hkv, D]); c.k_cache / c.v_cache are then the [NB, Hkv, 16, D]
    permuted views.  alibi: per-query-head ALiBi slopes (the reference includes the bias)."""
    assert len(lens) == S
    g = torch.Generator().manual_seed(seed)
    c = Case()
    c.S, c.Hq, c.Hkv, c.D, c.lens = S, Hq, Hkv, D, list(lens)
    c.dtype, c.fp8 = dtype, fp8
    c.k_scale = float(k_scale) if np.ndim(k_scale) == 0 else np.asarray(k_scale, dtype=np.float32)
    c.v_scale = float(v_scale) if np.ndim(v_scale) == 0 else np.asarray(v_scale, dtype=np.float32)
    c.alibi = None if alibi is None else np.asarray(alibi, dtype=np.float32)
    c.scale = 1.0 / math.sqrt(D)
    nb = [(L + B - 1) // B for L in lens]
    c.NB = sum(nb) + extra_blocks
    c.maxNB = max(nb + [1]) + 2
    p = torch.randperm(c.NB, generator=g) if perm is None else torch.as_tensor(perm)
    bt = torch.full((S, c.maxNB), table_pad, dtype=torch.int32)
    o = 0
    for s in range(S):
        bt[s, :nb[s]] = p[o:o + nb[s]].to(torch.int32)
        o += nb[s]
    c.block_table = bt
    c.seq_lens = torch.tensor(lens, dtype=torch.int32)
    c.q = torch.randn(S, Hq, D, generator=g).to(dtype)
    kv_dt = torch.bfloat16 if fp8 else dtype   # an E4M3 cache is written from bf16 rows
    c.K = [(torch.randn(L, Hkv, D, generator=g) * kv_sigma).to(kv_dt) for L in lens]
    c.V = [(torch.randn(L, Hkv, D, generator=g) * kv_sigma).to(kv_dt) for L in lens]
    cdt = torch.uint8 if fp8 else dtype
    shape = (c.NB, B, Hkv, D) if nhd else (c.NB, Hkv, B, D)
    kb, vb = torch.empty(shape, dtype=cdt), torch.empty(shape, dtype=cdt)
    kb.view(torch.uint8).fill_(0xFF)   # NaN everywhere nothing is written
    vb.view(torch.uint8).fill_(0xFF)
    c.k_cache = kb.permute(0, 2, 1, 3) if nhd else kb
    c.v_cache = vb.permute(0, 2, 1, 3) if nhd else vb
    c.Kval, c.Vval = [], []
    for s, L in enumerate(lens):
        if L == 0:
            c.Kval.append(np.zeros((0, Hkv, D)))
            c.Vval.append(np.zeros((0, Hkv, D)))
            continue
        t = torch.arange(L)
        blk = bt[s][t // B].long()
        off = t % B
        if fp8:
            ck = np.zeros((L, Hkv, D), dtype=np.uint8)
            cv = np.zeros((L, Hkv, D), dtype=np.uint8)
            oracle.write_flat(bf16_bits(c.K[s]), "bf16", np.arange(L), ck, "e4m3", k_scale)
            oracle.write_flat(bf16_bits(c.V[s]), "bf16", np.arange(L), cv, "e4m3", v_scale)
            c.k_cache[blk, :, off, :] = torch.from_numpy(ck)
            c.v_cache[blk, :, off, :] = torch.from_numpy(cv)
            c.Kval.append(oracle.cache_values(ck, "e4m3", k_scale))
            c.Vval.append(oracle.cache_values(cv, "e4m3", v_scale))
        else:
            c.k_cache[blk, :, off, :] = c.K[s]
            c.v_cache[blk, :, off, :] = c.V[s]
            c.Kval.append(c.K[s].double().numpy())
            c.Vval.append(c.V[s].double().numpy())
    return c


def reference(c: Case) -> np.ndarray:
    qd = c.q.double().numpy()
    out = np.zeros((c.S, c.Hq, c.D))
    for s in range(c.S):
        if c.alibi is not None:
            if c.lens[s] > 0:
                out[s] = oracle.attention_causal(qd[s][None], c.Kval[s], c.Vval[s], c.scale, c.alibi)[0]
        else:
            out[s] = oracle.dense_decode(qd[s], c.Kval[s], c.Vval[s], c.scale)
    return out


class OnGpu:
    pass


def to_gpu(c: Case, device="cuda") -> OnGpu:
    g = OnGpu()
    for name in ("q", "block_table", "seq_lens"):
        setattr(g, name, getattr(c, name).to(device))
    for name in ("k_cache", "v_cache"):   # keep the layout (an NHD view stays a view of NHD storage)
        t = getattr(c, name)
        base = t.permute(0, 2, 1, 3).contiguous().to(device) if t.stride(2) > t.stride(1) else t.contiguous().to(device)
        setattr(g, name, base.permute(0, 2, 1, 3) if t.stride(2) > t.stride(1) else base)
    g.out = torch.empty_like(g.q)
    g.k_scale = torch.tensor(np.atleast_1d(c.k_scale), dtype=torch.float32, device=device)
    g.v_scale = torch.tensor(np.atleast_1d(c.v_scale), dtype=torch.float32, device=device)
    g.scale_stride = 0 if np.ndim(c.k_scale) == 0 else 1
    g.alibi = None if c.alibi is None else torch.tensor(c.alibi, dtype=torch.float32, device=device)
    g.err = torch.zeros(1, dtype=torch.int32, device=device)
    g.ws = torch.zeros(64 << 20, dtype=torch.uint8, device=device)   # zero before first use
    return g


def run(c: Case, g: OnGpu, partition_size=0, out=None) -> torch.Tensor:
    import paged_decode_attention_reshape_gb300 as pa
    o = g.out if out is None else out
    if out is None:
        o.fill_(float("nan"))   # every output must be written by this call
    if g.scale_stride == 0 and g.alibi is None:
        pa.pa_decode_ex(o, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, c.scale, c.Hkv,
                        g.k_scale if c.fp8 else None, g.v_scale if c.fp8 else None, partition_size, g.ws, g.err)
    else:
        pa.pa_decode_opt(o, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, c.scale, c.Hkv,
                         g.k_scale if c.fp8 else None, g.v_scale if c.fp8 else None, g.scale_stride, g.alibi,
                         partition_size, g.ws, g.err)
    return o
