"""Paged decode on the GPU, through the C ABI, against the fp64 oracle.

Bar: |gpu - oracle| <= 1e-3 + 1 bf16 ulp of the oracle value, element by element;
split-KV results within the same bar of the unsplit ones."""
import numpy as np
import pytest
import torch

from gpu_cases import assert_close, make_case, reference, run, to_gpu

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu

LENS = [0, 1, 15, 16, 17, 33, 100, 257, 700, 1100]   # empty, single token, ragged tails, several tiles
PARTS = [-1, 16, 64, 512, 0, -2, -4, -8, -100]       # unsplit, splits of 1/4/32 pages, heuristic,
                                                      # cluster splits into 2/4/8 equal parts, balanced


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


SHAPES = [
    # (Hq, Hkv, D, q dtype, fp8 cache)
    (32, 8, 64, torch.bfloat16, False),
    (32, 8, 128, torch.bfloat16, False),
    (4, 4, 128, torch.bfloat16, False),     # MHA: one query head per KV head
    (32, 2, 128, torch.bfloat16, False),    # G = 16: two 8-head groups per KV head
    (8, 2, 256, torch.bfloat16, False),
    (16, 2, 64, torch.float16, False),
    (12, 4, 128, torch.float16, False),     # G = 3: partial head group
    (64, 8, 128, torch.bfloat16, True),     # E4M3 cache, G = 8
    (8, 1, 128, torch.float16, True),
    (16, 4, 256, torch.bfloat16, True),
    (4, 4, 64, torch.float32, False),       # fp32 CUDA-core path
    (32, 8, 128, torch.float32, False),
    (16, 2, 256, torch.float32, False),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "Hq%d_Hkv%d_D%d_%s%s" % (
    s[0], s[1], s[2], str(s[3]).split(".")[-1], "_e4m3" if s[4] else ""))
def test_decode_matches_oracle(shape):
    Hq, Hkv, D, dt, fp8 = shape
    c = make_case(len(LENS), Hq, Hkv, D, LENS, dtype=dt, fp8=fp8, seed=D + Hq,
                  k_scale=0.05 if fp8 else 1.0, v_scale=0.07 if fp8 else 1.0)
    ref = reference(c)
    g = to_gpu(c)
    outs = {}
    for P in PARTS:
        out = run(c, g, P).clone()
        torch.cuda.synchronize()
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == 0, (P, rc, bits)
        got = out.double().cpu().numpy()
        assert not np.isnan(got).any(), P
        assert_close(got, ref, "partition %d" % P)
        outs[P] = got
    for P in PARTS[1:]:
        assert_close(outs[P], outs[-1].astype(np.float64), "split %d vs unsplit" % P)


def test_physical_permutation_does_not_change_the_result():
    """Same logical K/V under different block permutations: bit-identical outputs."""
    lens = [40, 300, 17, 129]
    outs = []
    for perm_seed in range(3):
        nb = sum((L + 15) // 16 for L in lens) + 5
        perm = torch.randperm(nb, generator=torch.Generator().manual_seed(100 + perm_seed))
        c = make_case(4, 32, 8, 128, lens, seed=5, perm=perm)
        g = to_gpu(c)
        outs.append([run(c, g, P).clone().cpu() for P in (-1, 64, -4)])
    for o in outs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(o, outs[0]))


def test_in_place_output_over_q():
    lens = [5, 100, 333]
    for P in (-1, 32, -4):
        c = make_case(3, 16, 4, 128, lens, seed=11)
        g = to_gpu(c)
        ref_out = run(c, g, P).clone()
        run(c, g, P, out=g.q)          # out is q
        torch.cuda.synchronize()
        assert torch.equal(g.q, ref_out), P


def test_default_entry_point_with_internal_workspace():
    """pa_decode (no _ex): library-held workspace, heuristic partitions (splits here)."""
    lens = [3000, 5000]
    c = make_case(2, 32, 8, 128, lens, seed=3)
    g = to_gpu(c)
    P, n = pa.pa_decode_plan(2, 32, 8, 128, c.maxNB, pa.PA_BF16, 0, 0)
    assert P > 0 and n > 1
    pa.pa_decode(g.out, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, c.scale, c.Hkv)
    torch.cuda.synchronize()
    assert_close(g.out.double().cpu().numpy(), reference(c), "pa_decode")


def test_partition_example_1100_tokens():
    """The pages' 1100-token sequence at 512-token partitions (3 partitions, the last with
    5 blocks, partly valid), against the oracle and the unsplit path."""
    c = make_case(1, 8, 2, 128, [1100], seed=1100)
    g = to_gpu(c)
    ref = reference(c)
    a = run(c, g, 512).double().cpu().numpy()
    b = run(c, g, -1).double().cpu().numpy()
    assert_close(a, ref, "P=512")
    assert_close(a, b, "P=512 vs unsplit")


def test_block_id_out_of_range_is_reported_not_faulted():
    c = make_case(3, 8, 2, 128, [40, 64, 20], seed=9)
    c.block_table[1, 2] = c.NB + 7        # inside the sequence's first ceil(64/16) = 4 blocks
    c.block_table[2, 0] = -3
    g = to_gpu(c)
    for P in (-1, 16, -2):
        run(c, g, P)
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == -6, (rc, bits)
        assert bits & pa.PA_DEVERR_BLOCK_RANGE
    # sequence 0 (valid table row) is still computed correctly in the unsplit path
    out = run(c, g, -1).double().cpu().numpy()
    pa.pa_check_device_error(g.err)
    assert_close(out[0], reference(c)[0], "valid row next to bad rows")


def test_seq_len_beyond_table_is_reported():
    c = make_case(2, 8, 2, 64, [40, 20], seed=2)
    c.seq_lens[1] = c.maxNB * 16 + 1
    g = to_gpu(c)
    run(c, g, -1)
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == -6 and bits & pa.PA_DEVERR_SEQLEN_RANGE


def _checked(c, g, P, out=None):
    o = run(c, g, P, out=out)
    torch.cuda.synchronize()
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == 0, (P, rc, bits)
    return o.double().cpu().numpy()


BAL = pa.PA_PARTITION_BALANCED


@pytest.mark.parametrize("lens", [
    [0, 0, 0],                                   # nothing to read: all-zero rows
    [1, 0, 17],                                  # 3 pages in all, fewer than the CTAs of a row
    [5000] + [1] * 40 + [0, 0, 0] + [300],       # one long sequence over many CTAs, many 1-page ones
    [16] * 57 + [2000, 15, 0, 33],               # boundaries on page edges, several sequences per CTA
], ids=["all_empty", "fewer_pages_than_ctas", "long_and_short", "many_per_cta"])
def test_balanced_split_edges(lens):
    c = make_case(len(lens), 32, 8, 128, lens, seed=len(lens) * 7 + 1)
    ref = reference(c)
    g = to_gpu(c)
    g.out.fill_(float("nan"))
    got = _checked(c, g, BAL)
    assert_close(got, ref, "balanced")
    assert_close(got, _checked(c, g, -1), "balanced vs unsplit")


def test_balanced_split_largest_batch_and_limit():
    rng = np.random.default_rng(511)
    lens = rng.integers(0, 200, size=511).tolist()
    c = make_case(511, 8, 2, 64, lens, seed=511)
    g = to_gpu(c)
    assert_close(_checked(c, g, BAL), reference(c), "511 sequences")
    c2 = make_case(512, 8, 2, 64, [1] * 512, seed=512)
    g2 = to_gpu(c2)
    with pytest.raises(pa.PAError) as e:
        run(c2, g2, BAL)
    assert e.value.status == -7


def test_balanced_split_repeats_and_recovers_after_errors():
    """The arrival counters return to zero after every call, after calls with a bad block id
    or a bad length too: the same workspace then gives the right result again."""
    lens = [700, 33, 1500, 2, 260]
    for fp8 in (False, True):
        c = make_case(5, 64 if fp8 else 32, 8, 128, lens, fp8=fp8, seed=77, k_scale=0.05, v_scale=0.05)
        ref = reference(c)
        g = to_gpu(c)
        outs = [_checked(c, g, BAL) for _ in range(3)]
        for o in outs:
            assert_close(o, ref, "repeat fp8=%s" % fp8)
        assert all(np.array_equal(outs[0], o) for o in outs[1:])
        good_bt, good_sl = g.block_table.clone(), g.seq_lens.clone()
        g.block_table[2, 40] = c.NB + 3
        run(c, g, BAL)
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == -6 and bits & pa.PA_DEVERR_BLOCK_RANGE
        g.block_table.copy_(good_bt)
        g.seq_lens[1] = c.maxNB * 16 + 1
        run(c, g, BAL)
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == -6 and bits & pa.PA_DEVERR_SEQLEN_RANGE
        g.seq_lens.copy_(good_sl)
        assert_close(_checked(c, g, BAL), ref, "after errors fp8=%s" % fp8)
