"""The five workloads at full size, staged exactly as bench.py stages them
(NaN-poisoned pool, history written through the library, then one measured
step: cache write + decode with the default partition plan), against the oracle.

c1, c2, c3 and c4 are compared in full (every sequence and query head; c4 at
each partition size of its sweep), c5 on 64 of its 128 sequences with all 64
query heads; the oracle computes each sequence from its regenerated logical K/V,
never through the block table, so a CTA that read another sequence's or head's
pages would show.  Split is compared against unsplit everywhere, and the
variants on sampled outputs.  Cache writes are compared bit for bit."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import bench
import oracle
from gpu_cases import assert_close
from workloads import configs, data

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu
B = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


def _bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_heads(w, s, heads):
    """fp64 oracle outputs [len(heads), D] of sequence s for the given query heads."""
    kvh = sorted({h // w.G for h in heads})
    K, V = data.logical_kv(w, s, kv_heads=kvh)
    if w.kv_dtype == "e4m3":
        L = K.shape[0]
        ck = np.zeros((L, len(kvh), w.D), dtype=np.uint8)
        cv = np.zeros((L, len(kvh), w.D), dtype=np.uint8)
        ksc = w.k_scales() if np.ndim(w.k_scales()) == 0 else np.asarray(w.k_scales())[kvh]
        vsc = w.v_scales() if np.ndim(w.v_scales()) == 0 else np.asarray(w.v_scales())[kvh]
        oracle.write_flat(_bits16(K), "bf16", np.arange(L), ck, "e4m3", ksc)
        oracle.write_flat(_bits16(V), "bf16", np.arange(L), cv, "e4m3", vsc)
        Kv = oracle.cache_values(ck, "e4m3", ksc)
        Vv = oracle.cache_values(cv, "e4m3", vsc)
    else:
        Kv, Vv = K.double().numpy(), V.double().numpy()
    q = data.q(w, "cpu")[s].double().numpy()
    out = []
    for h in heads:
        j = kvh.index(h // w.G)
        if w.alibi is not None:
            out.append(oracle.attention_causal(q[h][None, None], Kv[:, j:j + 1], Vv[:, j:j + 1], w.scale,
                                               w.alibi[h:h + 1])[0, 0])
        else:
            out.append(oracle.dense_decode(q[h][None], Kv[:, j:j + 1], Vv[:, j:j + 1], w.scale)[0])
    return np.stack(out)


def oracle_all_heads(w, seqs):
    """fp64 oracle outputs [len(seqs), Hq, D] of every query head of the given sequences,
    one sequence per task on the host cores (the oracle's C calls release the GIL)."""
    n = max(1, min(16, len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(n) as ex:
        return np.stack(list(ex.map(lambda s: oracle_heads(w, int(s), range(w.Hq)), seqs)))


def oracle_rows(w, s, heads):
    """fp64 oracle outputs [nq, len(heads), D] of sequence s's query tokens (varlen workloads)."""
    kvh = sorted({h // w.G for h in heads})
    K, V = data.logical_kv(w, s, kv_heads=kvh)
    Kv, Vv = K.double().numpy(), V.double().numpy()
    q = data.q(w, "cpu").double().numpy()[s * w.nq:(s + 1) * w.nq]
    out = []
    for h in heads:
        j = kvh.index(h // w.G)
        out.append(oracle.attention_causal(q[:, h:h + 1], Kv[:, j:j + 1], Vv[:, j:j + 1], w.scale)[:, 0])
    return np.stack(out, axis=1)


def step(st, P=0):
    Pp, _, ws = bench.workspace_for(st, P)
    bench.run_write(st)
    bench.run_decode(st, P, ws)
    torch.cuda.synchronize()
    rc, bits = pa.pa_check_device_error(st.err)
    assert rc == 0, (rc, bits)
    return st.out.double().cpu().numpy()


def check_step_write(st, rows=None):
    """Cache rows at the step's slots (bit for bit) against the oracle's flat write of the step rows."""
    w = st.w
    valid = np.nonzero(w.step_slot >= 0)[0]
    if rows is not None:
        valid = valid[rows]
    slots = torch.as_tensor(w.step_slot[valid])
    blk, off = slots // B, slots % B
    for cache, src, scale in ((st.k_cache, st.k_step, w.k_scales()), (st.v_cache, st.v_step, w.v_scales())):
        got = cache[blk.cuda(), :, off.cuda(), :].cpu()             # [n, Hkv, D]
        rows_in = src[torch.as_tensor(valid).cuda()].cpu()
        n = len(valid)
        if w.cache_dtype == "e4m3":
            ref = np.zeros((n, w.Hkv, w.D), dtype=np.uint8)
            oracle.write_flat(_bits16(rows_in), "bf16", np.arange(n), ref, "e4m3", scale)
            assert np.array_equal(got.numpy(), ref)
        elif w.cache_dtype == "bf16":
            ref = np.zeros((n, w.Hkv, w.D), dtype=np.uint16)
            oracle.write_flat(_bits16(rows_in), "bf16", np.arange(n), ref, "bf16")
            assert np.array_equal(_bits16(got), ref)
        else:
            ref = np.zeros((n, w.Hkv, w.D), dtype=np.float32)
            oracle.write_flat(rows_in.numpy(), "f32", np.arange(n), ref, "f32")
            assert np.array_equal(got.numpy().view(np.uint32), ref.view(np.uint32))


def test_c1_full():
    w = configs.get("c1")
    st = bench.stage(w)
    for P in (0, -1, 16, 32):
        got = step(st, P)
        check_step_write(st)
        for s in range(w.S):
            assert_close(got[s], oracle_heads(w, s, range(w.Hq)), "c1 seq %d P=%d" % (s, P))
    # the padding row (slot -1, NaN data) wrote nothing: the pool holds no NaN where a
    # sequence lives, and the rest of the pool is still the NaN poison
    kc = st.k_cache.cpu()
    used = {int(b) for s in range(w.S) for b in w.block_table[s][:w.n_blocks_of(s)]}
    for b in range(w.num_blocks):
        if b in used:
            continue
        assert torch.isnan(kc[b]).all()


def test_c2_full():
    w = configs.get("c2")
    st = bench.stage(w)
    got = step(st, 0)
    check_step_write(st)
    for s in range(w.S):
        assert_close(got[s], oracle_heads(w, s, range(w.Hq)), "c2 seq %d" % s)


def test_c3_full():
    """Every (sequence, query head) output of the 256-sequence batch against the oracle."""
    w = configs.get("c3")
    st = bench.stage(w)
    got = step(st, 0)
    check_step_write(st)
    ref = oracle_all_heads(w, range(w.S))
    for s in range(w.S):
        assert_close(got[s], ref[s], "c3 seq %d" % s)


def test_c4_full_over_partition_sizes():
    w = configs.get("c4")
    st = bench.stage(w)
    outs = {P: step(st, P) for P in (0, 128, 256, 512, 1024, 2048, 4096, -1)}
    ref = oracle_all_heads(w, range(w.S))   # every head, the +20 outlier heads among them
    for s in range(w.S):
        for P, got in outs.items():
            assert_close(got[s], ref[s], "c4 seq %d P=%d" % (s, P))
    for P, got in outs.items():
        assert_close(got, outs[-1], "c4 split %d vs unsplit" % P)


def test_c5_fp8_write_and_sampled_decode():
    w = configs.get("c5")
    st = bench.stage(w)
    got = step(st, 0)
    rng = np.random.default_rng(55)
    nvalid = int((w.step_slot >= 0).sum())
    check_step_write(st, rows=np.sort(rng.choice(nvalid, size=512, replace=False)))
    # padding rows (slot -1) wrote nothing: their positions still hold the history values
    pad = np.nonzero(w.step_slot < 0)[0]
    assert len(pad) == w.notes["padding_rows"] > 0
    for s in np.unique(w.step_seq[pad]):
        pos = w.step_pos[pad][w.step_seq[pad] == s]
        K, V = data.history_rows(w, int(s), "cpu", positions=torch.as_tensor(pos))
        slots = torch.as_tensor(w.slot_of(int(s), pos))
        for cache, rows_in, scale in ((st.k_cache, K, w.k_scale), (st.v_cache, V, w.v_scale)):
            ref = np.zeros((len(pos), w.Hkv, w.D), dtype=np.uint8)
            oracle.write_flat(_bits16(rows_in), "bf16", np.arange(len(pos)), ref, "e4m3", scale)
            gotc = cache[(slots // B).cuda(), :, (slots % B).cuda(), :].cpu().numpy()
            assert np.array_equal(gotc, ref)
    seqs = np.sort(rng.choice(w.S, size=64, replace=False))   # 64 sequences, every query head
    ref = oracle_all_heads(w, seqs)
    for i, s in enumerate(seqs):
        assert_close(got[s], ref[i], "c5 seq %d" % s)
    # split (the plan) against unsplit on every output
    assert_close(got, step(st, -1), "c5 split vs unsplit")


def test_c5_step_equals_two_calls():
    """c5 through pa_decode_step (8192 new rows: the write on the grid it gets beside an early-
    reading decode, many tokens per thread) against the write and the decode called one after
    the other (checked against the oracle above): both caches and every output bit for bit."""
    w = configs.get("c5")
    a, b = bench.stage(w), bench.stage(w)
    assert isinstance(b.new_rows_start, torch.Tensor)  # pa_decode_step with early reads
    _, _, ws_a = bench.workspace_for(a, 0)
    _, _, ws_b = bench.workspace_for(b, 0)
    bench.run_write(a)
    bench.run_decode(a, 0, ws_a)
    bench.run_step(b, 0, ws_b)
    torch.cuda.synchronize()
    for st in (a, b):
        rc, bits = pa.pa_check_device_error(st.err)
        assert rc == 0, (rc, bits)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.k_cache.view(torch.uint8), b.k_cache.view(torch.uint8))
    assert torch.equal(a.v_cache.view(torch.uint8), b.v_cache.view(torch.uint8))


# ---------------------------------------- variants: NHD layout, ALiBi, per-head scales

def test_c2_nhd_full_and_equal_to_hnd():
    """c2's values in the NHD cache layout: every output against the oracle, and bit-identical
    to the HND run (same pages, same arithmetic)."""
    w = configs.get("c2-nhd")
    st = bench.stage(w)
    got = step(st, 0)
    check_step_write(st)
    for s in range(w.S):
        assert_close(got[s], oracle_heads(w, s, range(w.Hq)), "c2-nhd seq %d" % s)
    hnd = bench.stage(configs.get("c2"))
    assert np.array_equal(got, step(hnd, 0))


def test_c3_alibi_sampled():
    w = configs.get("c3-alibi")
    st = bench.stage(w)
    got = step(st, 0)
    rng = np.random.default_rng(34)
    for s in rng.choice(w.S, size=6, replace=False):
        heads = sorted(rng.choice(w.Hq, size=4, replace=False).tolist())
        assert_close(got[s][heads], oracle_heads(w, int(s), heads), "c3-alibi seq %d" % s)


def test_c5_heads_write_and_sampled_decode():
    w = configs.get("c5-heads")
    st = bench.stage(w)
    got = step(st, 0)
    rng = np.random.default_rng(56)
    nvalid = int((w.step_slot >= 0).sum())
    check_step_write(st, rows=np.sort(rng.choice(nvalid, size=512, replace=False)))
    for s in rng.choice(w.S, size=6, replace=False):
        heads = sorted(rng.choice(w.Hq, size=3, replace=False).tolist())
        assert_close(got[s][heads], oracle_heads(w, int(s), heads), "c5-heads seq %d" % s)


def test_c3_spec4_write_and_sampled_varlen():
    """4 query tokens per sequence: the step writes each sequence's last 4 positions, and
    query i attends to the tokens up to its own position."""
    w = configs.get("c3-spec4")
    st = bench.stage(w)
    got = step(st, 0)
    check_step_write(st)
    rng = np.random.default_rng(35)
    for s in rng.choice(w.S, size=6, replace=False):
        heads = sorted(rng.choice(w.Hq, size=4, replace=False).tolist())
        ref = oracle_rows(w, int(s), heads)
        assert_close(got[s * w.nq:(s + 1) * w.nq][:, heads], ref, "c3-spec4 seq %d" % s)
    assert_close(got, step(st, -1), "plan vs unsplit")


def test_c3_chunk128_write_and_sampled_query_tile():
    """Chunked prefill at full size (256 sequences x 128 new tokens, 512 query rows per KV
    head, the query-tile tensor-core kernel): the step's write, sampled sequences and heads
    against the oracle, and the column-group path (fixed 4096-token partitions) on the same
    step to the same bar."""
    w = configs.get("c3-chunk128")
    assert w.query_tile()
    st = bench.stage(w)
    got = step(st, 0)
    rng = np.random.default_rng(128)
    nvalid = int((w.step_slot >= 0).sum())
    check_step_write(st, rows=np.sort(rng.choice(nvalid, size=512, replace=False)))
    for s in rng.choice(w.S, size=4, replace=False):
        heads = sorted(rng.choice(w.Hq, size=3, replace=False).tolist())
        ref = oracle_rows(w, int(s), heads)
        assert_close(got[s * w.nq:(s + 1) * w.nq][:, heads], ref, "c3-chunk128 seq %d" % s)
    assert_close(got, step(st, 4096), "query tile vs column groups")
