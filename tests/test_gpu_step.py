"""pa_decode_step (write + decode in one call, the decode reading untouched pages while the
write runs) against the same two operations called one after the other, and against the
oracle: outputs bit for bit, caches bit for bit, on single-token steps, chunk steps with
padding rows, FP8 caches with per-tensor and per-head scales, ALiBi, NHD caches and every
partition mode."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_close, make_case, reference, to_gpu

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


def _step_rows(c, nnew, seed, pad_frac=0.0):
    """New rows for each sequence's last nnew[s] positions (fresh values), their slots (a
    fraction set to -1: padding), and new_rows_start."""
    gen = torch.Generator().manual_seed(seed)
    rows, slots, start = [], [], [0]
    for s, L in enumerate(c.lens):
        n = nnew[s]
        for pos in range(L - n, L):
            slots.append(int(c.block_table[s, pos // 16]) * 16 + pos % 16)
        start.append(start[-1] + n)
    T = start[-1]
    K = torch.randn(T, c.Hkv, c.D, generator=gen).to(torch.bfloat16 if c.fp8 else c.dtype)
    V = torch.randn(T, c.Hkv, c.D, generator=gen).to(K.dtype)
    slots = np.array(slots, dtype=np.int64)
    if pad_frac > 0 and T:
        rng = np.random.default_rng(seed)
        slots[rng.random(T) < pad_frac] = -1
    return K, V, slots, np.array(start, dtype=np.int32)


def _two_calls(c, g, K, V, slots, P, ws, alibi, ks, vs, stride):
    kv = pa.PA_KV_FP8_E4M3 if c.fp8 else pa.PA_KV_AUTO
    pa.pa_reshape_and_cache_opt(K, V, g.k_cache, g.v_cache, slots, kv, ks, vs, stride, g.err)
    out = torch.full_like(g.q, float("nan"))
    pa.pa_decode_opt(out, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, c.scale, c.Hkv, ks, vs, stride,
                     alibi, P, ws, g.err)
    return out


CASES = [
    # (S, Hq, Hkv, D, lens, nnew, dtype, fp8, per-head scales, alibi, nhd, pad_frac)
    (8, 32, 8, 64, [1, 17, 300, 1100, 2000, 16, 33, 700], [1] * 8, torch.bfloat16, False, False, False, False, 0.0),
    (6, 32, 8, 128, [5, 64, 65, 500, 1500, 3000], [1] * 6, torch.bfloat16, False, False, True, True, 0.0),
    (5, 64, 8, 128, [70, 200, 1024, 1500, 4000], [64] * 5, torch.bfloat16, True, False, False, False, 0.05),
    (5, 64, 8, 128, [70, 200, 1024, 1500, 4000], [64] * 5, torch.bfloat16, True, True, False, False, 0.05),
    (4, 12, 4, 128, [1, 40, 900, 2500], [1, 3, 20, 40], torch.float16, False, False, False, False, 0.0),
]
IDS = ["decode_bf16_D64", "decode_bf16_D128_alibi_nhd", "chunk64_e4m3", "chunk64_e4m3_heads", "mixed_f16"]


@pytest.mark.parametrize("case", CASES, ids=IDS)
@pytest.mark.parametrize("P", [0, -1, 64, -2, pa.PA_PARTITION_BALANCED])
def test_step_equals_two_calls(case, P):
    S, Hq, Hkv, D, lens, nnew, dt, fp8, heads, alibi, nhd, pad = case
    ks = list(np.linspace(0.04, 0.075, Hkv).astype(np.float32)) if heads else (0.05 if fp8 else 1.0)
    vs = list(np.linspace(0.075, 0.04, Hkv).astype(np.float32)) if heads else (0.07 if fp8 else 1.0)
    slopes = list(2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)) if alibi else None
    c = make_case(S, Hq, Hkv, D, lens, dtype=dt, fp8=fp8, seed=S + D, k_scale=ks, v_scale=vs, alibi=slopes, nhd=nhd)
    K, V, slots, start = _step_rows(c, nnew, seed=D + S, pad_frac=pad)
    nrs = None if all(n == 1 for n in nnew) else torch.from_numpy(start).cuda()
    Kg, Vg, sg = K.cuda(), V.cuda(), torch.from_numpy(slots).cuda()
    ksg = torch.tensor(np.atleast_1d(ks), dtype=torch.float32, device="cuda") if fp8 else None
    vsg = torch.tensor(np.atleast_1d(vs), dtype=torch.float32, device="cuda") if fp8 else None
    stride = 1 if heads else 0
    al = None if slopes is None else torch.tensor(slopes, dtype=torch.float32, device="cuda")
    need = max(pa.pa_decode_workspace_size(S, Hq, Hkv, D, c.maxNB, x) for x in (64, pa.PA_PARTITION_BALANCED))
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    # the two calls
    g1 = to_gpu(c)
    ref_out = _two_calls(c, g1, Kg, Vg, sg, P, ws, al, ksg, vsg, stride)
    torch.cuda.synchronize()
    assert pa.pa_check_device_error(g1.err) == (0, 0)
    # one call
    g2 = to_gpu(c)
    out = torch.full_like(g2.q, float("nan"))
    pa.pa_decode_step(out, g2.q, Kg, Vg, g2.k_cache, g2.v_cache, sg, g2.block_table, g2.seq_lens, c.scale, Hkv,
                      new_rows_start=nrs, k_scale=ksg, v_scale=vsg, scale_stride=stride, alibi_slopes=al,
                      partition_size=P, workspace=ws, device_error=g2.err)
    torch.cuda.synchronize()
    assert pa.pa_check_device_error(g2.err) == (0, 0)
    assert torch.equal(out.view(torch.int16) if out.dtype != torch.float32 else out, ref_out.view(torch.int16)
                       if ref_out.dtype != torch.float32 else ref_out)
    assert torch.equal(g2.k_cache.contiguous().view(torch.uint8), g1.k_cache.contiguous().view(torch.uint8))
    assert torch.equal(g2.v_cache.contiguous().view(torch.uint8), g1.v_cache.contiguous().view(torch.uint8))


def test_step_against_the_oracle():
    """A single-token bf16 step: the output against the fp64 oracle over the history plus
    the new rows (the oracle never reads through the block table)."""
    S, Hq, Hkv, D = 6, 32, 8, 128
    lens = [1, 30, 257, 1000, 1600, 64]
    c = make_case(S, Hq, Hkv, D, lens, seed=91)
    K, V, slots, _ = _step_rows(c, [1] * S, seed=92)
    # the oracle's logical K/V with the new rows in place
    for s, L in enumerate(lens):
        c.Kval[s][L - 1] = K[s].double().numpy()
        c.Vval[s][L - 1] = V[s].double().numpy()
    g = to_gpu(c)
    out = torch.full_like(g.q, float("nan"))
    pa.pa_decode_step(out, g.q, K.cuda(), V.cuda(), g.k_cache, g.v_cache, torch.from_numpy(slots).cuda(),
                      g.block_table, g.seq_lens, c.scale, Hkv, device_error=g.err)
    torch.cuda.synchronize()
    assert pa.pa_check_device_error(g.err) == (0, 0)
    assert_close(out.double().cpu().numpy(), reference(c), "pa_decode_step vs oracle")


def test_step_validates_before_launching():
    """A decode-side argument error leaves the cache untouched (nothing was launched)."""
    c = make_case(2, 8, 2, 64, [10, 20], seed=5)
    g = to_gpu(c)
    K, V, slots, _ = _step_rows(c, [1, 1], seed=6)
    before = g.k_cache.clone()
    bad_out = torch.empty(2, 8, 32, dtype=torch.bfloat16, device="cuda")  # wrong head size
    with pytest.raises(pa.PAError):
        pa.pa_decode_step(bad_out, g.q, K.cuda(), V.cuda(), g.k_cache, g.v_cache, torch.from_numpy(slots).cuda(),
                          g.block_table, g.seq_lens, c.scale, 2, device_error=g.err)
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), g.k_cache.view(torch.int16))  # bits (the pool holds NaN)
