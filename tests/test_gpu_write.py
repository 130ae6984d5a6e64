"""The cache write on the GPU, through the C ABI, against the oracle's flat-slot
write: bit-exact, including E4M3 quantisation; negative slots write nothing."""
import numpy as np
import pytest
import torch

from gpu_cases import bf16_bits

import oracle
import paged_decode_attention_reshape_gb300 as pa

pytestmark = pytest.mark.gpu
B = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    pa.lib()
    torch.cuda.set_device(0)


def flat_view(cache: torch.Tensor) -> np.ndarray:
    """[NB, Hkv, 16, D] HND cache -> [NB*16, Hkv, D] indexed by slot = block*16 + offset (raw bytes)."""
    NB, H, _, D = cache.shape
    c = cache.cpu().permute(0, 2, 1, 3).reshape(NB * B, H, D).contiguous()
    return c.view(torch.uint8).numpy().reshape(NB * B, H, -1)


def np_bytes(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint8).reshape(a.shape[0], a.shape[1], -1)


def run_write(key, value, slots, NB, cache_dtype, kv_mode, k_scale=1.0, v_scale=1.0, poison=True):
    dev = "cuda"
    H, D = key.shape[1], key.shape[2]
    kc = torch.empty((NB, H, B, D), dtype=cache_dtype, device=dev)
    vc = torch.empty((NB, H, B, D), dtype=cache_dtype, device=dev)
    fill = 0xFF if poison else 0
    kc.view(torch.uint8).fill_(fill)
    vc.view(torch.uint8).fill_(fill)
    ks = torch.tensor([k_scale], dtype=torch.float32, device=dev)
    vs = torch.tensor([v_scale], dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pa.pa_reshape_and_cache(key.to(dev), value.to(dev), kc, vc, torch.as_tensor(slots, dtype=torch.int64).to(dev),
                            kv_mode, ks, vs, err)
    rc, bits = pa.pa_check_device_error(err)
    return kc, vc, rc, bits


def oracle_write(rows_np, rows_dt, slots, NB, cache_np_dtype, cache_dt, scale=1.0, poison=True):
    T, H, D = rows_np.shape
    flat = np.full((NB * B, H, D), 0xFF if poison else 0, dtype=np.uint8).view(cache_np_dtype) \
        if cache_np_dtype == np.uint8 else None
    if flat is None:
        width = np.dtype(cache_np_dtype).itemsize
        flat = np.full((NB * B, H, D * width), 0xFF if poison else 0, dtype=np.uint8).view(cache_np_dtype)
    oracle.write_flat(rows_np, rows_dt, np.asarray(slots, dtype=np.int64), flat, cache_dt, scale)
    return flat


@pytest.mark.parametrize("dtype,ddt,npdt", [(torch.float32, "f32", np.float32), (torch.bfloat16, "bf16", np.uint16),
                                            (torch.float16, "f16", np.uint16)])
def test_copy_write_bit_exact_with_padding_rows(dtype, ddt, npdt):
    g = torch.Generator().manual_seed(1)
    T, H, D, NB = 300, 8, 128, 64
    key = torch.randn(T, H, D, generator=g).to(dtype)
    val = torch.randn(T, H, D, generator=g).to(dtype)
    slots = torch.randperm(NB * B, generator=g)[:T].to(torch.int64)
    pad = torch.randperm(T, generator=g)[:25]
    slots[pad] = -1
    key[pad] = float("nan")        # padding rows carry NaN: must never land anywhere
    val[pad] = float("nan")
    kc, vc, rc, bits = run_write(key, val, slots, NB, dtype, pa.PA_KV_AUTO)
    assert rc == 0, bits
    kn = key.view(torch.int32 if dtype == torch.float32 else torch.int16).numpy().view(npdt)
    vn = val.view(torch.int32 if dtype == torch.float32 else torch.int16).numpy().view(npdt)
    ref_k = oracle_write(kn, ddt, slots.numpy(), NB, npdt, ddt)
    ref_v = oracle_write(vn, ddt, slots.numpy(), NB, npdt, ddt)
    assert np.array_equal(flat_view(kc), np_bytes(ref_k))
    assert np.array_equal(flat_view(vc), np_bytes(ref_v))


def test_worked_example_slot_36():
    """block_table [7, 2, 9], position 20 -> slot 36 = block 2, offset 4."""
    H, D, NB = 2, 64, 16
    key = torch.randn(1, H, D).to(torch.bfloat16)
    val = torch.randn(1, H, D).to(torch.bfloat16)
    kc, vc, rc, _ = run_write(key, val, [36], NB, torch.bfloat16, pa.PA_KV_AUTO, poison=False)
    assert rc == 0
    assert torch.equal(kc[2, :, 4, :].cpu(), key[0]) and torch.equal(vc[2, :, 4, :].cpu(), val[0])
    kc[2, :, 4, :] = 0
    assert not kc.view(torch.int16).any()


@pytest.mark.parametrize("scales", [(0.05, 0.05), (1.0, 0.37), (3.0, 0.0078125)])
def test_fp8_write_every_bf16_value(scales):
    """All 65536 bf16 bit patterns through the E4M3 write, K and V with their own scales."""
    ks, vs = scales
    bits = np.arange(65536, dtype=np.uint16).reshape(64, 8, 128)
    rng = np.random.default_rng(3)
    vbits = rng.permutation(bits.reshape(-1)).reshape(64, 8, 128)
    key = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    val = torch.from_numpy(vbits.view(np.int16).copy()).view(torch.bfloat16)
    NB = 8
    slots = np.arange(64)
    kc, vc, rc, _ = run_write(key, val, slots, NB, torch.uint8, pa.PA_KV_FP8_E4M3, ks, vs)
    assert rc == 0
    ref_k = oracle_write(bits, "bf16", slots, NB, np.uint8, "e4m3", ks)
    ref_v = oracle_write(vbits, "bf16", slots, NB, np.uint8, "e4m3", vs)
    for got, ref, src in ((flat_view(kc), ref_k, bits), (flat_view(vc), ref_v, vbits)):
        got = got[:64]
        ref = ref[:64]
        x = (src.astype(np.uint32) << 16).view(np.float32)
        nan_in = np.isnan(x)
        # NaN inputs: the pages say nothing; both sides must give an E4M3 NaN code
        assert np.all((got[nan_in] & 0x7F) == 0x7F) and np.all((ref[nan_in] & 0x7F) == 0x7F)
        assert np.array_equal(got[~nan_in], ref[~nan_in])


def test_fp8_write_fp32_rows_near_rounding_midpoints():
    mags = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2.0
    sc = np.float32(0.05)
    base = (mids * float(sc)).astype(np.float32)
    xs = [base]
    for _ in range(3):
        xs.append(np.nextafter(xs[-1], np.float32(np.inf)))
    lo = [base]
    for _ in range(3):
        lo.append(np.nextafter(lo[-1], np.float32(0)))
    x = np.concatenate(xs + lo[1:])
    x = np.concatenate([x, -x])
    n = (x.size + 127) // 128 * 128
    x = np.concatenate([x, np.zeros(n - x.size, dtype=np.float32)]).reshape(-1, 1, 128)
    T = x.shape[0]
    key = torch.from_numpy(x.copy())
    kc, vc, rc, _ = run_write(key, key.clone(), np.arange(T), (T + 15) // 16, torch.uint8, pa.PA_KV_FP8_E4M3,
                              0.05, 0.05)
    assert rc == 0
    ref = oracle_write(x, "f32", np.arange(T), (T + 15) // 16, np.uint8, "e4m3", 0.05)
    assert np.array_equal(flat_view(kc)[:T], ref[:T])


def test_strided_views_fused_qkv_and_combined_kv():
    """key/value as views of a fused [T, 3, H, D] projection; K/V caches as views of one
    [NB, 2, H, 16, D] tensor."""
    g = torch.Generator().manual_seed(4)
    T, H, D, NB = 50, 4, 64, 16
    qkv = torch.randn(T, 3, H, D, generator=g).to(torch.bfloat16).cuda()
    key, val = qkv[:, 1], qkv[:, 2]
    kv = torch.zeros((NB, 2, H, B, D), dtype=torch.bfloat16, device="cuda")
    kc, vc = kv[:, 0], kv[:, 1]
    slots = torch.randperm(NB * B, generator=g)[:T].to(torch.int64).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(key, val, kc, vc, slots, pa.PA_KV_AUTO, None, None, err)
    assert pa.pa_check_device_error(err)[0] == 0
    s = slots.cpu()
    blk, off = s // B, s % B
    assert torch.equal(kv[blk, 0, :, off, :].cpu(), key.cpu())
    assert torch.equal(kv[blk, 1, :, off, :].cpu(), val.cpu())


def test_out_of_range_slot_is_reported_and_writes_nothing():
    H, D, NB = 2, 64, 4
    key = torch.randn(3, H, D).to(torch.bfloat16)
    kc, vc, rc, bits = run_write(key, key.clone(), [5, NB * B, NB * B + 1000], NB, torch.bfloat16, pa.PA_KV_AUTO,
                                 poison=False)
    assert rc == -6 and bits & pa.PA_DEVERR_SLOT_RANGE
    assert torch.equal(kc[0, :, 5, :].cpu(), key[0])
    kc[0, :, 5, :] = 0
    assert not kc.view(torch.int16).any()


def test_empty_write_is_a_no_op():
    kc = torch.zeros((2, 2, B, 64), dtype=torch.bfloat16, device="cuda")
    e = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    pa.pa_reshape_and_cache(e, e, kc, kc.clone(), torch.empty(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert not kc.view(torch.int16).any()


@pytest.mark.parametrize("scales", ["tensor", "heads", "odd"])
@pytest.mark.parametrize("in_dt", ["bf16", "f16"])
@pytest.mark.parametrize("H,D", [(8, 128), (2, 64), (24, 256)], ids=["8x128", "2x64", "24x256"])
def test_fp8_write_all_16bit_patterns(H, D, in_dt, scales):
    """Every bf16 / f16 bit pattern (zeros, subnormals, infinities, NaN, magnitudes beyond
    2^80 and below 2^-80 among them) through the E4M3 write, bit for bit against the oracle:
    token shapes that fit one block of threads and wider ones, one scale per tensor, one per
    KV head, or unusual ones (a negative scale; a scale below 2^-40, which takes the IEEE
    division), padding rows skipped."""
    per_head = scales == "heads"
    rng = np.random.default_rng(H * 1000 + D)
    n = H * D
    T = (65536 + n - 1) // n + 3
    pats = np.zeros(T * n, dtype=np.uint16)
    pats[:65536] = rng.permutation(65536).astype(np.uint16)
    kbits = pats.reshape(T, H, D)
    vbits = rng.permutation(pats).reshape(T, H, D)
    tdt = torch.bfloat16 if in_dt == "bf16" else torch.float16
    key = torch.from_numpy(kbits.view(np.int16).copy()).view(tdt)
    val = torch.from_numpy(vbits.view(np.int16).copy()).view(tdt)
    NB = (T + 15) // 16 + 2
    slots = rng.permutation(NB * B)[:T].astype(np.int64)
    pad = rng.choice(T, size=2, replace=False)
    slots[pad] = -1
    if scales == "heads":
        ks = (0.05 * (1 + np.arange(H) / 8)).astype(np.float32)
        vs = (0.9 / (1 + np.arange(H))).astype(np.float32)
    elif scales == "odd":
        ks, vs = np.float32(-0.05), np.float32(2.0 ** -45)
    else:
        ks, vs = np.float32(0.05), np.float32(3.0)
    dev = "cuda"
    kc = torch.full((NB, H, B, D), 0xFF, dtype=torch.uint8, device=dev)
    vc = torch.full((NB, H, B, D), 0xFF, dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pa.pa_reshape_and_cache_opt(key.to(dev), val.to(dev), kc, vc, torch.from_numpy(slots).to(dev),
                                pa.PA_KV_FP8_E4M3, torch.tensor(np.atleast_1d(ks), device=dev),
                                torch.tensor(np.atleast_1d(vs), device=dev), 1 if per_head else 0, err)
    rc, bits = pa.pa_check_device_error(err)
    assert rc == 0, bits
    for cache, src, sc in ((kc, kbits, ks), (vc, vbits, vs)):
        ref = oracle_write(src, in_dt, slots, NB, np.uint8, "e4m3", sc)
        got = flat_view(cache)
        x = (src.astype(np.uint32) << 16).view(np.float32) if in_dt == "bf16" else src.view(np.float16)
        nan_rows = np.isnan(x)
        written = slots[slots >= 0]
        rows = np.nonzero(slots >= 0)[0]
        g, r = got[written], ref[written]
        nan_in = nan_rows[rows]
        assert np.all((g[nan_in] & 0x7F) == 0x7F) and np.all((r[nan_in] & 0x7F) == 0x7F)
        assert np.array_equal(g[~nan_in], r[~nan_in])
        untouched = np.setdiff1d(np.arange(NB * B), written)
        assert np.all(got[untouched] == 0xFF)
