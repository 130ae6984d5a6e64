"""pa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory where they run attention (a plugin that is handed only its input
and output buffers, or a serving loop whose free memory all belongs to its
KV-cache pool).  Its split-KV scratch is a fixed buffer inside the library.

Checks, through the C ABI: its output matches the fp64 oracle and pa_decode_ex (the
entry point with a caller workspace) within the parity tolerance, on two calls in a
row and after a call of another shape has left its data in the shared buffer; a
problem that needs more scratch than the buffer holds is refused with
PA_ERR_WORKSPACE; a call with a bad argument is refused before anything runs.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

from gpu_cases import assert_close, make_case, reference, run, to_gpu

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


def _noalloc(c, g, partition_size):
    out = torch.full_like(g.q, float("nan"))   # every output must be written by the call
    pa.pa_decode_noalloc(out, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, c.scale, c.Hkv,
                         g.k_scale if c.fp8 else None, g.v_scale if c.fp8 else None, partition_size, g.err)
    torch.cuda.synchronize()
    rc, bits = pa.pa_check_device_error(g.err)
    assert rc == 0, (rc, bits)
    return out.double().cpu().numpy()


def test_matches_workspace_entry_point_on_consecutive_calls():
    cases = [
        (make_case(3, 32, 8, 128, [3000, 5000, 700], seed=21), 512),             # bf16, split
        (make_case(4, 64, 8, 128, [1500, 4100, 60, 2222], fp8=True, seed=22,     # e4m3 cache, G = 8
                   k_scale=0.05, v_scale=0.05), 1024),
        (make_case(2, 8, 2, 64, [33, 900], seed=23), -1),                        # unsplit: no scratch used
        (make_case(2, 64, 8, 128, [30000, 9000], dtype=torch.float16, fp8=True,  # f16 query, e4m3 cache,
                   seed=24, k_scale=0.05, v_scale=0.05), 0),                      # the library's own plan
    ]
    for c, P in cases:
        g = to_gpu(c)
        oracle_out = reference(c)
        ref = run(c, g, P).double().cpu().numpy()
        assert_close(ref, oracle_out, "pa_decode_ex, P=%d" % P)
        first = _noalloc(c, g, P)
        second = _noalloc(c, g, P)
        assert_close(first, oracle_out, "first no-alloc call against the oracle, P=%d" % P)
        assert_close(second, oracle_out, "second no-alloc call against the oracle, P=%d" % P)
        assert_close(first, ref, "first no-alloc call, P=%d" % P)
        assert_close(second, ref, "second no-alloc call, P=%d" % P)
    # the first shape again, after the others left their partial results in the buffer
    c, P = cases[0]
    g = to_gpu(c)
    assert_close(_noalloc(c, g, P), run(c, g, P).double().cpu().numpy(), "after other shapes")


def test_refuses_problems_larger_than_the_scratch_buffer():
    S, Hq, Hkv, D, MB = 64, 64, 8, 256, 8192
    need = pa.pa_decode_workspace_size(S, Hq, Hkv, D, MB, 256)
    assert need > pa.PA_NOALLOC_SCRATCH_BYTES
    dev = "cuda"
    q = torch.zeros(S, Hq, D, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(4, Hkv, 16, D, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(S, MB, dtype=torch.int32, device=dev)
    sl = torch.ones(S, dtype=torch.int32, device=dev)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_noalloc(torch.empty_like(q), q, kc, kc.clone(), bt, sl, 0.1, Hkv, partition_size=256)
    assert e.value.status == -4
    # the same problem unsplit needs no scratch and runs
    pa.pa_decode_noalloc(torch.empty_like(q), q, kc, kc.clone(), bt, sl, 0.1, Hkv, partition_size=-1)
    torch.cuda.synchronize()


def test_bad_argument_is_refused_before_anything_runs():
    """Every argument is checked before the scratch is touched: a call with an output of the
    wrong type is refused, and a good call right after it is still correct."""
    c = make_case(3, 32, 8, 128, [3000, 5000, 700], seed=25)
    g = to_gpu(c)
    bad_out = torch.empty(g.q.shape, dtype=torch.float16, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_noalloc(bad_out, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, c.scale, c.Hkv,
                             partition_size=512, device_error=g.err)
    assert e.value.status == -1
    bad_lens = g.seq_lens.to(torch.int64)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_noalloc(g.out, g.q, g.k_cache, g.v_cache, g.block_table, bad_lens, c.scale, c.Hkv,
                             partition_size=512, device_error=g.err)
    assert e.value.status == -2
    assert_close(_noalloc(c, g, 512), reference(c), "good call after refused ones")
