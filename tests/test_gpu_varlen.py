"""pa_attention_varlen on the GPU, through the C ABI, against the fp64 oracle: several new
query tokens per sequence (speculative decoding, chunked prefill), causal within the
sequence, on every kernel and partition mode.

Bar: |gpu - oracle| <= 1e-3 + 1 bf16 ulp of the oracle value, element by element."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_close, make_case

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu

PARTS = [-1, 64, 0, -2]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


class Varlen:
    pass


def make_varlen(lens, nqs, Hq, Hkv, D, dtype=torch.bfloat16, fp8=False, seed=0, alibi=None, nq_max=None, nhd=False):
    """Caches for sequences of visible length lens[s] (history + new tokens), nqs[s] new query
    tokens each, packed in q [sum(nqs), Hq, D]."""
    c = make_case(len(lens), Hq, Hkv, D, lens, dtype=dtype, fp8=fp8, seed=seed,
                  k_scale=0.05 if fp8 else 1.0, v_scale=0.07 if fp8 else 1.0, alibi=alibi, nhd=nhd)
    v = Varlen()
    v.c = c
    v.nqs = list(nqs)
    v.qsl = np.concatenate([[0], np.cumsum(nqs)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed + 1000)
    v.q = torch.randn(int(v.qsl[-1]), Hq, D, generator=g).to(dtype)
    v.nq_max = max(nqs + [1]) if nq_max is None else nq_max
    return v


def reference(v):
    c = v.c
    out = np.zeros((v.q.shape[0], c.Hq, c.D))
    qd = v.q.double().numpy()
    for s in range(c.S):
        a, b = int(v.qsl[s]), int(v.qsl[s + 1])
        if b > a:
            out[a:b] = oracle.attention_causal(qd[a:b], c.Kval[s], c.Vval[s], c.scale, c.alibi)
    return out


def on_gpu(v):
    c = v.c
    g = Varlen()
    g.q = v.q.cuda()
    g.qsl = torch.from_numpy(v.qsl).cuda()
    g.k_cache, g.v_cache = c.k_cache.cuda(), c.v_cache.cuda()
    g.bt, g.sl = c.block_table.cuda(), c.seq_lens.cuda()
    g.ks = torch.tensor([c.k_scale], dtype=torch.float32, device="cuda")
    g.vs = torch.tensor([c.v_scale], dtype=torch.float32, device="cuda")
    g.alibi = None if c.alibi is None else torch.from_numpy(c.alibi).cuda()
    g.err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # split-KV workspace as documented: the decode size with num_heads = Hq * max_query_len
    need = max(pa.pa_decode_workspace_size(c.S, c.Hq * v.nq_max, c.Hkv, c.D, c.maxNB, P) for P in (64, 16))
    g.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    return g


def run(v, g, P, out=None):
    c = v.c
    o = torch.full_like(g.q, float("nan")) if out is None else out
    pa.pa_attention_varlen(o, g.q, g.k_cache, g.v_cache, g.qsl, g.bt, g.sl, c.scale, c.Hkv, v.nq_max,
                           k_scale=g.ks if c.fp8 else None, v_scale=g.vs if c.fp8 else None,
                           alibi_slopes=g.alibi, partition_size=P, workspace=g.ws, device_error=g.err)
    return o


SHAPES = [
    # (Hq, Hkv, D, q dtype, fp8 cache)
    (32, 8, 64, torch.bfloat16, False),     # G = 4: 2 query tokens per 8-column group
    (32, 8, 128, torch.bfloat16, False),
    (64, 8, 128, torch.bfloat16, True),     # G = 8: one token per group
    (12, 4, 128, torch.float16, False),     # G = 3: groups cut tokens apart
    (4, 4, 64, torch.bfloat16, False),      # MHA: 8 tokens per group
    (32, 2, 128, torch.bfloat16, False),    # G = 16: two groups per token
    (8, 2, 128, torch.float32, False),      # fp32 CUDA-core path
]
IDS = ["Hq%d_Hkv%d_D%d_%s%s" % (s[0], s[1], s[2], str(s[3]).split(".")[-1], "_e4m3" if s[4] else "")
       for s in SHAPES]
LENS = [1, 17, 100, 700, 1100, 40, 0]
NQS = [1, 5, 8, 3, 16, 40, 0]   # whole prompt (seq 0 and 5), chunks, an empty query


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_varlen_matches_oracle(shape):
    Hq, Hkv, D, dt, fp8 = shape
    v = make_varlen(LENS, NQS, Hq, Hkv, D, dtype=dt, fp8=fp8, seed=Hq + D)
    ref = reference(v)
    g = on_gpu(v)
    outs = {}
    for P in PARTS:
        got = run(v, g, P)
        torch.cuda.synchronize()
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == 0, (P, rc, bits)
        got = got.double().cpu().numpy()
        assert not np.isnan(got).any(), P
        assert_close(got, ref, "varlen partition %d" % P)
        outs[P] = got
    for P in PARTS[1:]:
        assert_close(outs[P], outs[-1], "split %d vs unsplit" % P)


@pytest.mark.parametrize("shape", SHAPES[:3], ids=IDS[:3])
def test_varlen_alibi(shape):
    Hq, Hkv, D, dt, fp8 = shape
    slopes = 2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)
    v = make_varlen(LENS, NQS, Hq, Hkv, D, dtype=dt, fp8=fp8, seed=7 * D, alibi=slopes)
    ref = reference(v)
    g = on_gpu(v)
    for P in PARTS:
        got = run(v, g, P)
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == 0, (P, rc, bits)
        assert_close(got.double().cpu().numpy(), ref, "varlen alibi partition %d" % P)


def test_one_token_per_sequence_is_decode_bit_for_bit():
    lens = [1, 33, 500, 1100, 2]
    v = make_varlen(lens, [1] * len(lens), 32, 8, 128, seed=11)
    g = on_gpu(v)
    c = v.c
    dec = torch.empty_like(g.q)
    for P in (-1, 64, -2):
        pa.pa_decode_ex(dec, g.q, g.k_cache, g.v_cache, g.bt, g.sl, c.scale, c.Hkv, None, None, P, g.ws, g.err)
        assert torch.equal(run(v, g, P), dec), P


def test_larger_max_query_len_and_spec_decode_batch():
    """max_query_len above every n_s (more, empty column groups); a spec-decode batch of
    4-token queries over long histories."""
    lens = [300, 1500, 64, 2000]
    v = make_varlen(lens, [4, 4, 4, 4], 32, 8, 128, seed=21, nq_max=9)
    g = on_gpu(v)
    ref = reference(v)
    for P in PARTS:
        got = run(v, g, P)
        assert pa.pa_check_device_error(g.err) == (0, 0)
        assert_close(got.double().cpu().numpy(), ref, "nq_max 9, partition %d" % P)


def test_bad_query_ranges_are_reported_and_skipped():
    lens = [50, 40, 30]
    v = make_varlen(lens, [3, 5, 2], 16, 4, 64, seed=31, nq_max=4)   # sequence 1 has more than nq_max
    g = on_gpu(v)
    ref = reference(v)
    got = run(v, g, -1)
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == -6 and bits & pa.PA_DEVERR_SEQLEN_RANGE
    got = got.double().cpu().numpy()
    a1, b1 = int(v.qsl[1]), int(v.qsl[2])
    assert np.isnan(got[a1:b1]).all()                    # nothing written for sequence 1
    assert_close(got[:a1], ref[:a1], "sequence 0")
    assert_close(got[b1:], ref[b1:], "sequence 2")
    # a query range past the packed rows, and more queries than visible tokens
    g.qsl = torch.tensor([0, 3, 7, 12], dtype=torch.int32, device="cuda")   # rows 7..11 > Tq = 10
    v.nq_max = 5
    run(v, g, -1)
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == -6 and bits & pa.PA_DEVERR_SEQLEN_RANGE
    g.qsl = torch.tensor([0, 3, 3, 10], dtype=torch.int32, device="cuda")
    g.sl = torch.tensor([50, 40, 6], dtype=torch.int32, device="cuda")     # 7 queries, 6 visible tokens
    v.nq_max = 7
    run(v, g, -1)
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == -6 and bits & pa.PA_DEVERR_SEQLEN_RANGE


def test_host_side_refusals():
    v = make_varlen([20], [2], 8, 2, 64, seed=41)
    g = on_gpu(v)
    with pytest.raises(pa.PAError) as e:
        run(v, g, pa.PA_PARTITION_BALANCED)
    assert e.value.status == -7
    v.nq_max = 0
    with pytest.raises(pa.PAError) as e:
        run(v, g, -1)
    assert e.value.status == -1


CHUNK_SHAPES = [
    # (Hq, Hkv, D, q dtype, alibi): query-tile kernel (>= 32 query columns per KV head)
    (32, 8, 128, torch.bfloat16, False),
    (32, 8, 64, torch.float16, False),
    (8, 8, 128, torch.bfloat16, True),      # MHA: one row per query token
    (40, 8, 128, torch.bfloat16, True),     # G = 5: 64-row tiles cut tokens apart
]


@pytest.mark.parametrize("shape", CHUNK_SHAPES,
                         ids=["Hq%d_Hkv%d_D%d_%s%s" % (s[0], s[1], s[2], str(s[3]).split(".")[-1],
                                                       "_alibi" if s[4] else "") for s in CHUNK_SHAPES])
def test_long_chunks_match_oracle(shape):
    """Chunked prefill: up to 192 new tokens over histories of up to 2100 tokens (many
    64-row query tiles, ragged last tile and page); the same result unsplit, by the
    heuristic and split into 64-token partitions (the column-group kernels)."""
    Hq, Hkv, D, dt, alibi = shape
    slopes = 2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq) if alibi else None
    lens, nqs = [1200, 700, 2100, 64, 5], [192, 100, 64, 64, 1]
    v = make_varlen(lens, nqs, Hq, Hkv, D, dtype=dt, seed=3 * Hq + D, alibi=slopes)
    ref = reference(v)
    g = on_gpu(v)
    outs = {}
    for P in (-1, 0, 64):
        got = run(v, g, P)
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == 0, (P, rc, bits)
        outs[P] = got.clone()
        got = got.double().cpu().numpy()
        assert not np.isnan(got).any(), P
        assert_close(got, ref, "chunk partition %d" % P)
    assert torch.equal(outs[0], outs[-1])
    assert_close(outs[64].double().cpu().numpy(), outs[-1].double().cpu().numpy(), "split 64 vs unsplit")


def test_query_tile_at_32_columns_head_size_64():
    """Head size 64 switches to the query tile at 32 query columns per KV head (8 new tokens x
    G = 4): one partly filled 128-row tile per KV head, against the oracle and against the
    column-group kernels (a split asked for)."""
    lens, nqs = [300, 129, 40, 1000, 8], [8, 8, 5, 8, 8]
    v = make_varlen(lens, nqs, 32, 8, 64, seed=51)
    assert v.nq_max * 4 == 32
    ref = reference(v)
    g = on_gpu(v)
    outs = {}
    for P in (-1, 64):
        got = run(v, g, P)
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == 0, (P, rc, bits)
        outs[P] = got.double().cpu().numpy()
        assert not np.isnan(outs[P]).any(), P
        assert_close(outs[P], ref, "32 columns, partition %d" % P)
    assert_close(outs[64], outs[-1], "column groups vs query tile")


def test_query_tile_bad_ranges_are_reported_and_skipped():
    lens = [50, 40, 30]
    v = make_varlen(lens, [3, 17, 2], 32, 8, 64, seed=33, nq_max=16)  # 64 columns; sequence 1 > nq_max
    g = on_gpu(v)
    ref = reference(v)
    got = run(v, g, -1)
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == -6 and bits & pa.PA_DEVERR_SEQLEN_RANGE
    got = got.double().cpu().numpy()
    a1, b1 = int(v.qsl[1]), int(v.qsl[2])
    assert np.isnan(got[a1:b1]).all()
    assert_close(got[:a1], ref[:a1], "sequence 0")
    assert_close(got[b1:], ref[b1:], "sequence 2")
