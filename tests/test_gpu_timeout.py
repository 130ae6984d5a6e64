"""The bounded pipeline waits, made to run out on purpose through the `first_wait_limit`
option (a wait limit of zero polls on the first K/V wait), on the GPU, through the C ABI.

A wait that gives up must not leave the GPU in a bad state or write anything wrong: the
kernel waits (with the normal limit) for the copies it had in flight, sets
PA_DEVERR_WAIT_TIMEOUT in the device error word, writes no output for its work item -- nor
for a split-KV unit any of whose parts gave up -- and returns.  The checks here: the call
reports PA_ERR_DEVICE_TIMEOUT with the timeout bit, the NaN-filled output is left untouched,
and the next call with the normal limit, on the same workspace, matches the fp64 oracle
(the split-KV arrival counters are back at zero).  A one-poll limit, which may or may not
run out, gives outputs that are each either untouched or correct.

Failures come from the library's own bounded waits: no fault, trap or endless loop is used
("vLLM 源码完全拆解（七）", 正确性不变量与调试方法: a failure must surface, not corrupt
results silently)."""
import numpy as np
import pytest
import torch

from gpu_cases import assert_close, make_case, reference, to_gpu, within_tol
from test_gpu_varlen import make_varlen, on_gpu
from test_gpu_varlen import reference as varlen_reference

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu
TIMEOUT = -8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


def _decode(c, g, P, limit):
    out = torch.full_like(g.q, float("nan"))
    pa.pa_decode_opt(out, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, c.scale, c.Hkv,
                     g.k_scale if c.fp8 else None, g.v_scale if c.fp8 else None, 0, None, P, g.ws, g.err,
                     first_wait_limit=limit)
    torch.cuda.synchronize()
    rc, bits = pa.pa_check_device_error(g.err)
    return rc, bits, out.double().cpu().numpy()


CASES = {
    "bf16_d128": dict(S=3, Hq=32, Hkv=8, D=128, lens=[3000, 700, 1500], seed=801),
    "bf16_d64": dict(S=4, Hq=32, Hkv=8, D=64, lens=[2048, 33, 900, 1], seed=802),
    "fp8_d128": dict(S=2, Hq=64, Hkv=8, D=128, lens=[4100, 2222], fp8=True, k_scale=0.05, v_scale=0.05, seed=803),
}


@pytest.mark.parametrize("P", [-1, 512, pa.PA_PARTITION_BALANCED, -2], ids=["unsplit", "p512", "balanced", "cluster2"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_wait_that_runs_out_writes_nothing_and_recovers(name, P):
    c = make_case(**CASES[name])
    g = to_gpu(c)
    ref = reference(c)
    for _ in range(2):   # twice in a row: the counters must be back at zero after a timed-out call
        rc, bits, got = _decode(c, g, P, -1)
        assert rc == TIMEOUT and bits == pa.PA_DEVERR_WAIT_TIMEOUT, (rc, bits)
        assert np.isnan(got).all(), "a timed-out call wrote output"
    rc, bits, got = _decode(c, g, P, 0)
    assert rc == 0, (rc, bits)
    assert_close(got, ref, "%s P=%d after timeouts" % (name, P))


@pytest.mark.parametrize("P", [-1, 256])
def test_decode_one_poll_limit_gives_untouched_or_correct_rows(P):
    c = make_case(**CASES["bf16_d128"])
    g = to_gpu(c)
    ref = reference(c)
    rc, bits, got = _decode(c, g, P, 1)
    assert rc in (0, TIMEOUT) and bits in (0, pa.PA_DEVERR_WAIT_TIMEOUT), (rc, bits)
    for s in range(c.S):
        for h in range(c.Hq):
            row = got[s, h]
            assert np.isnan(row).all() or within_tol(row, ref[s, h]).all(), (s, h)
    rc, bits, got = _decode(c, g, P, 0)
    assert rc == 0, (rc, bits)
    assert_close(got, ref, "after the one-poll call")


@pytest.mark.parametrize("D", [128, 64])
def test_query_tile_wait_that_runs_out_writes_nothing_and_recovers(D):
    """pa_attention_varlen on the tcgen05 query-tile kernel (>= 64 query columns per KV head, 32 at D = 64):
    the MMA issuer's first K/V-group wait gives up, every role leaves, the copies and MMAs in
    flight are waited for, the tensor memory is freed, nothing is written."""
    v = make_varlen([700, 300, 129], [128, 40, 129], 32, 8, D, seed=900 + D)
    g = on_gpu(v)
    c = v.c

    def call(limit):
        out = torch.full_like(g.q, float("nan"))
        pa.pa_attention_varlen(out, g.q, g.k_cache, g.v_cache, g.qsl, g.bt, g.sl, c.scale, c.Hkv, v.nq_max,
                               partition_size=0, workspace=g.ws, device_error=g.err, first_wait_limit=limit)
        torch.cuda.synchronize()
        rc, bits = pa.pa_check_device_error(g.err)
        return rc, bits, out.double().cpu().numpy()

    for _ in range(2):
        rc, bits, got = call(-1)
        assert rc == TIMEOUT and bits == pa.PA_DEVERR_WAIT_TIMEOUT, (rc, bits)
        assert np.isnan(got).all(), "a timed-out query-tile call wrote output"
    rc, bits, got = call(0)
    assert rc == 0, (rc, bits)
    assert_close(got, varlen_reference(v), "query tile D=%d after timeouts" % D)


def test_decode_step_wait_that_runs_out_still_writes_the_cache():
    """pa_decode_step: the cache write has no pipeline wait and lands; the decode's first wait
    gives up and writes nothing; a normal step after it is correct."""
    c = make_case(**CASES["bf16_d64"])
    g = to_gpu(c)
    S = c.S
    # the step's rows: each sequence's newest position, written again with the same values
    last = [L - 1 for L in c.lens]
    slots = torch.tensor([int(c.block_table[s, last[s] // 16]) * 16 + last[s] % 16 for s in range(S)],
                         dtype=torch.int64, device="cuda")
    key = torch.stack([c.K[s][last[s]] for s in range(S)]).cuda()
    val = torch.stack([c.V[s][last[s]] for s in range(S)]).cuda()
    ref = reference(c)
    for limit, expect in ((-1, TIMEOUT), (0, 0)):
        out = torch.full_like(g.q, float("nan"))
        pa.pa_decode_step(out, g.q, key, val, g.k_cache, g.v_cache, slots, g.block_table, g.seq_lens, c.scale,
                          c.Hkv, device_error=g.err, first_wait_limit=limit)
        torch.cuda.synchronize()
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == expect, (limit, rc, bits)
        got = out.double().cpu().numpy()
        if expect:
            assert np.isnan(got).all()
        else:
            assert_close(got, ref, "step after a timed-out step")
