"""The _opt entry points on the GPU, through the C ABI, against the fp64 oracle:
per-head FP8 scales (write and decode), the NHD cache layout (write and decode) and
ALiBi (decode, on every kernel and partition mode).

Writes are compared bit for bit; decode within 1e-3 + 1 bf16 ulp of the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import assert_close, make_case, reference, run, to_gpu

import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu

PARTS = [-1, 64, 0, -2, pa.PA_PARTITION_BALANCED]
LENS = [0, 1, 17, 100, 700, 1100]
HEAD_SCALES = np.array([0.05, 0.37, 1.0, 3.0], dtype=np.float32)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


def _bits(t: torch.Tensor, tag: str) -> np.ndarray:
    if tag == "f32":
        return t.contiguous().numpy()
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _scale_array(stride: int) -> np.ndarray:
    """Per-head scales laid out at h * stride (NaN in between, so a wrong index shows);
    stride 0: one shared scale."""
    if stride == 0:
        return np.array([0.37], dtype=np.float32)
    a = np.full(len(HEAD_SCALES) * stride, np.nan, dtype=np.float32)
    a[::stride] = HEAD_SCALES
    return a


# --------------------------------------------------------------------- write

@pytest.mark.parametrize("stride", [0, 1, 3])
@pytest.mark.parametrize("layout", ["hnd", "nhd"])
@pytest.mark.parametrize("in_dt,tag", [(torch.bfloat16, "bf16"), (torch.float16, "f16"), (torch.float32, "f32")],
                         ids=["bf16", "f16", "f32"])
def test_write_e4m3_per_head_scales_and_layout(in_dt, tag, layout, stride):
    T, Hkv, D, NB = 37, 4, 128, 12
    g = torch.Generator().manual_seed(T + stride + (7 if layout == "nhd" else 0))
    key = (torch.randn(T, Hkv, D, generator=g) * 3).to(in_dt)
    value = (torch.randn(T, Hkv, D, generator=g) * 2).to(in_dt)
    slots = torch.randperm(NB * 16, generator=g)[:T].long()
    slots[[3, 10]] = -1
    shape = (NB, 16, Hkv, D) if layout == "nhd" else (NB, Hkv, 16, D)
    kb = torch.full(shape, 0xFF, dtype=torch.uint8, device="cuda")
    vb = torch.full(shape, 0xFF, dtype=torch.uint8, device="cuda")
    kv, vv = (kb.permute(0, 2, 1, 3), vb.permute(0, 2, 1, 3)) if layout == "nhd" else (kb, vb)
    sc = torch.from_numpy(_scale_array(stride)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache_opt(key.cuda(), value.cuda(), kv, vv, slots.cuda(), pa.PA_KV_FP8_E4M3,
                                k_scale=sc, v_scale=sc, scale_stride=stride, device_error=err)
    assert pa.pa_check_device_error(err) == (0, 0)
    head = float(_scale_array(0)[0]) if stride == 0 else HEAD_SCALES
    for src, got in ((key, kv), (value, vv)):
        ref = np.full((NB * 16, Hkv, D), 0xFF, dtype=np.uint8)
        oracle.write_flat(_bits(src, tag), tag, slots.numpy(), ref, "e4m3", head)
        flat = got.permute(0, 2, 1, 3).reshape(NB * 16, Hkv, D).cpu().numpy()
        assert np.array_equal(flat, ref)


@pytest.mark.parametrize("layout", ["hnd", "nhd"])
def test_write_copy_layouts_and_shared_scale_matches_plain_entry(layout):
    T, Hkv, D, NB = 21, 8, 64, 6
    g = torch.Generator().manual_seed(5)
    key = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    value = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    slots = torch.randperm(NB * 16, generator=g)[:T].long()
    slots[0] = -1
    shape = (NB, 16, Hkv, D) if layout == "nhd" else (NB, Hkv, 16, D)
    kb = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vb = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    view = (lambda t: t.permute(0, 2, 1, 3)) if layout == "nhd" else (lambda t: t)
    pa.pa_reshape_and_cache_opt(key.cuda(), value.cuda(), view(kb), view(vb), slots.cuda())
    for src, got in ((key, kb), (value, vb)):
        ref = np.zeros((NB * 16, Hkv, D), dtype=np.uint16)
        oracle.write_flat(_bits(src, "bf16"), "bf16", slots.numpy(), ref, "bf16")
        flat = view(got).permute(0, 2, 1, 3).reshape(NB * 16, Hkv, D).cpu()
        assert np.array_equal(_bits(flat, "bf16"), ref)
    # FP8 with one shared scale: the _opt entry (stride 0) and the plain entry write the same bytes
    sc = torch.tensor([0.05], device="cuda")
    a = torch.zeros(NB, Hkv, 16, D, dtype=torch.uint8, device="cuda")
    b = torch.zeros_like(a)
    pa.pa_reshape_and_cache(key.cuda(), value.cuda(), a, a.clone(), slots.cuda(), pa.PA_KV_FP8_E4M3, sc, sc)
    pa.pa_reshape_and_cache_opt(key.cuda(), value.cuda(), b, b.clone(), slots.cuda(), pa.PA_KV_FP8_E4M3,
                                k_scale=sc, v_scale=sc, scale_stride=0)
    assert torch.equal(a, b)


# -------------------------------------------------------------------- decode

DECODE_SHAPES = [
    # (Hq, Hkv, D, q dtype, fp8 cache)
    (32, 8, 64, torch.bfloat16, False),
    (32, 8, 128, torch.bfloat16, False),
    (64, 8, 128, torch.bfloat16, True),
    (16, 4, 256, torch.float16, True),
    (12, 4, 128, torch.float16, False),
    (8, 2, 128, torch.float32, False),
]
IDS = ["Hq%d_Hkv%d_D%d_%s%s" % (s[0], s[1], s[2], str(s[3]).split(".")[-1], "_e4m3" if s[4] else "")
       for s in DECODE_SHAPES]


def _parts_match(c, g, ref, what):
    outs = {}
    for P in PARTS:
        out = run(c, g, P).clone()
        rc, bits = pa.pa_check_device_error(g.err)
        assert rc == 0, (what, P, rc, bits)
        got = out.double().cpu().numpy()
        assert_close(got, ref, "%s partition %d" % (what, P))
        outs[P] = got
    return outs


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=IDS)
def test_decode_nhd_layout_equals_hnd(shape):
    Hq, Hkv, D, dt, fp8 = shape
    kw = dict(dtype=dt, fp8=fp8, seed=D + Hq + 1, k_scale=0.05 if fp8 else 1.0, v_scale=0.07 if fp8 else 1.0)
    c_n = make_case(len(LENS), Hq, Hkv, D, LENS, nhd=True, **kw)
    c_h = make_case(len(LENS), Hq, Hkv, D, LENS, **kw)
    ref = reference(c_h)
    on = _parts_match(c_n, to_gpu(c_n), ref, "nhd")
    oh = _parts_match(c_h, to_gpu(c_h), ref, "hnd")
    for P in PARTS:   # same pages, same arithmetic: the layouts give identical outputs
        assert np.array_equal(on[P], oh[P]), P


@pytest.mark.parametrize("Hq,Hkv,D,dt", [(64, 8, 128, torch.bfloat16), (16, 4, 256, torch.float16),
                                         (8, 4, 128, torch.bfloat16)])
def test_decode_per_head_scales(Hq, Hkv, D, dt):
    ks = HEAD_SCALES[:Hkv] if Hkv <= 4 else np.resize(HEAD_SCALES, Hkv) * np.linspace(0.5, 1.5, Hkv).astype(np.float32)
    vs = ks[::-1].copy()
    c = make_case(len(LENS), Hq, Hkv, D, LENS, dtype=dt, fp8=True, seed=Hq * D, k_scale=ks, v_scale=vs)
    ref = reference(c)
    g = to_gpu(c)
    _parts_match(c, g, ref, "per-head scales")
    # the same scales at stride 2 (interleaved with NaN)
    g.k_scale = torch.tensor(np.stack([ks, np.full_like(ks, np.nan)], 1).ravel(), device="cuda")
    g.v_scale = torch.tensor(np.stack([vs, np.full_like(vs, np.nan)], 1).ravel(), device="cuda")
    g.scale_stride = 2
    _parts_match(c, g, ref, "per-head scales, stride 2")


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=IDS)
def test_decode_alibi(shape):
    Hq, Hkv, D, dt, fp8 = shape
    slopes = 2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)        # the usual geometric ALiBi slopes
    c = make_case(len(LENS), Hq, Hkv, D, LENS, dtype=dt, fp8=fp8, seed=3 * D + Hq, alibi=slopes,
                  k_scale=0.05 if fp8 else 1.0, v_scale=0.07 if fp8 else 1.0)
    ref = reference(c)
    _parts_match(c, to_gpu(c), ref, "alibi")
