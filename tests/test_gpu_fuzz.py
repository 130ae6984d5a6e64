"""Randomised decode and varlen cases on the GPU against the fp64 oracle: head counts, head
sizes, cache types, lengths (0 to a few thousand), layouts, per-head scales, ALiBi and every
partition mode drawn from a fixed seed.  Also the write + decode step captured in a CUDA graph
and replayed with new inputs."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_close, make_case, reference, run, to_gpu

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


def _draw(rng):
    D = int(rng.choice([64, 128, 256]))
    kind = rng.choice(["bf16", "f16", "e4m3", "f32"], p=[0.4, 0.2, 0.25, 0.15])
    if kind == "e4m3" and D == 64:
        D = 128
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    S = int(rng.integers(1, 12))
    lens = [int(x) for x in rng.integers(0, 2500, size=S)]
    if rng.random() < 0.3:
        lens[int(rng.integers(S))] = 0
    dt = {"bf16": torch.bfloat16, "f16": torch.float16, "e4m3": torch.bfloat16, "f32": torch.float32}[kind]
    fp8 = kind == "e4m3"
    ks = 0.05 if not fp8 or rng.random() < 0.5 else list(rng.uniform(0.03, 0.09, size=Hkv).astype(np.float32))
    vs = 0.07 if not isinstance(ks, list) else list(rng.uniform(0.03, 0.09, size=Hkv).astype(np.float32))
    alibi = list(2.0 ** (-8.0 * np.arange(1, Hkv * G + 1) / (Hkv * G))) if rng.random() < 0.3 else None
    nhd = bool(rng.random() < 0.3)
    P = int(rng.choice([-1, 0, 16, 64, 256, -2, -4, -8, pa.PA_PARTITION_BALANCED]))
    return dict(S=S, Hq=Hkv * G, Hkv=Hkv, D=D, lens=lens, dtype=dt, fp8=fp8, k_scale=ks if fp8 else 1.0,
                v_scale=vs if fp8 else 1.0, alibi=alibi, nhd=nhd), P


@pytest.mark.parametrize("seed", range(24))
def test_random_decode_cases(seed):
    rng = np.random.default_rng(1000 + seed)
    kw, P = _draw(rng)
    S, Hq, Hkv, D, lens = kw.pop("S"), kw.pop("Hq"), kw.pop("Hkv"), kw.pop("D"), kw.pop("lens")
    c = make_case(S, Hq, Hkv, D, lens, seed=seed, **kw)
    g = to_gpu(c)
    got = run(c, g, P).double().cpu().numpy()
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == 0, (rc, bits)
    assert_close(got, reference(c), "seed %d: S=%d Hq=%d Hkv=%d D=%d P=%d %s" % (seed, S, Hq, Hkv, D, P, kw))


def test_step_in_a_cuda_graph():
    """cache write + decode (split plan, caller workspace) captured once, replayed with new rows
    and queries copied into the captured input buffers."""
    S, Hq, Hkv, D = 6, 32, 8, 128
    lens = [700, 33, 1500, 1, 260, 90]
    c = make_case(S, Hq, Hkv, D, lens, seed=77)
    g = to_gpu(c)
    gen = torch.Generator().manual_seed(78)
    # the step writes each sequence's last position again (new values)
    slots = torch.tensor([int(c.block_table[s, (L - 1) // 16]) * 16 + (L - 1) % 16 for s, L in enumerate(lens)],
                         dtype=torch.int64, device="cuda")
    kin = torch.empty(S, Hkv, D, dtype=torch.bfloat16, device="cuda")
    vin = torch.empty_like(kin)
    ws = torch.zeros(pa.pa_decode_workspace_size(S, Hq, Hkv, D, c.maxNB, 64), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        pa.pa_reshape_and_cache(kin, vin, g.k_cache, g.v_cache, slots, stream=stream)
        pa.pa_decode_ex(g.out, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, c.scale, Hkv,
                        partition_size=64, workspace=ws, device_error=g.err, stream=stream)

    with torch.cuda.stream(stream):
        step()                                   # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for it in range(3):
        K = torch.randn(S, Hkv, D, generator=gen).to(torch.bfloat16)
        V = torch.randn(S, Hkv, D, generator=gen).to(torch.bfloat16)
        q = torch.randn(S, Hq, D, generator=gen).to(torch.bfloat16)
        kin.copy_(K)
        vin.copy_(V)
        g.q.copy_(q)
        graph.replay()
        torch.cuda.synchronize()
        assert pa.pa_check_device_error(g.err) == (0, 0)
        for s, L in enumerate(lens):
            c.Kval[s][L - 1] = K[s].double().numpy()
            c.Vval[s][L - 1] = V[s].double().numpy()
        c.q = q
        assert_close(g.out.double().cpu().numpy(), reference(c), "graph replay %d" % it)


def _draw_varlen(rng):
    """A varlen batch whose chunks reach both kernels: query columns per KV head (max new
    tokens x G) from a few (column groups) to several hundred (query tiles, one or two per CTA)."""
    D = int(rng.choice([64, 128]))
    dt = torch.bfloat16 if rng.random() < 0.7 else torch.float16
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 5, 8]))
    S = int(rng.integers(1, 5))
    long_chunks = rng.random() < 0.7
    cap = int(rng.choice([24, 48, 96])) if long_chunks else 6
    lens, nqs = [], []
    for _ in range(S):
        L = int(rng.integers(1, 1200))
        hi = min(L, cap)
        n = int(rng.integers(0, hi + 1))
        if long_chunks and rng.random() < 0.2:
            n = L  # a whole prompt
        lens.append(L)
        nqs.append(n)
    alibi = list(2.0 ** (-8.0 * np.arange(1, Hkv * G + 1) / (Hkv * G))) if rng.random() < 0.3 else None
    nhd = bool(rng.random() < 0.3)
    P = int(rng.choice([-1, 0, 64]))
    return dict(lens=lens, nqs=nqs, Hq=Hkv * G, Hkv=Hkv, D=D, dtype=dt, alibi=alibi, nhd=nhd), P


@pytest.mark.parametrize("seed", range(20))
def test_random_varlen_cases(seed):
    from test_gpu_varlen import make_varlen, on_gpu
    from test_gpu_varlen import reference as varlen_reference
    from test_gpu_varlen import run as varlen_run
    rng = np.random.default_rng(2000 + seed)
    kw, P = _draw_varlen(rng)
    v = make_varlen(kw["lens"], kw["nqs"], kw["Hq"], kw["Hkv"], kw["D"], dtype=kw["dtype"], seed=seed,
                    alibi=kw["alibi"], nhd=kw["nhd"])
    g = on_gpu(v)
    got = varlen_run(v, g, P)
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == 0, (rc, bits)
    got = got.double().cpu().numpy()
    assert not np.isnan(got).any()
    cols = max(kw["nqs"] + [1]) * (kw["Hq"] // kw["Hkv"])
    assert_close(got, varlen_reference(v), "seed %d: %s P=%d columns/KV head %d" % (seed, kw, P, cols))
