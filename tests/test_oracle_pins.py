"""Pins for the CPU oracle: each check ties it to something other than itself --
values the pages print, the OFP8 format table, a library routine (torch's
float8_e4m3fn conversion, scipy's softmax), closed forms and invariants.

CPU only (no GPU marker)."""
import math

import numpy as np
import pytest
import torch
from scipy.special import softmax

from conftest import golden_kv, golden_lines

import oracle

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ E4M3 codec

def test_e4m3_decode_matches_ofp8_table():
    for code, val in golden_lines("e4m3_values.txt"):
        got = oracle.e4m3_decode(np.array([int(code, 16)], dtype=np.uint8))[0]
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1.0, got) == math.copysign(1.0, float(val)), code


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decode_monotone_and_symmetric():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)


def _all_bf16_as_f32():
    bits = np.arange(65536, dtype=np.uint32) << 16
    return bits.view(np.float32)


def test_e4m3_encode_every_bf16_vs_torch():
    """RNE to E4M3 for every bf16 value; torch's (non-saturating) conversion is the
    library reference below 464, where the two definitions coincide."""
    x = _all_bf16_as_f32()
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    finite = np.isfinite(x) & (np.abs(x) < 464.0)
    assert np.array_equal(ours[finite], ref[finite])
    # saturation and NaN (the reading: satfinite, NaN -> 0x7F)
    big = np.isfinite(x) & (np.abs(x) >= 464.0) | np.isinf(x)
    assert np.all(ours[big & (x > 0)] == 0x7E) and np.all(ours[big & (x < 0)] == 0xFE)
    assert np.all(ours[np.isnan(x)] == 0x7F)


def test_e4m3_encode_ties_and_zero():
    # 2^-10 is halfway between 0 and the smallest subnormal: ties to even -> 0
    assert oracle.e4m3_encode(np.float32(2.0 ** -10)) == 0x00
    assert oracle.e4m3_encode(np.float32(-(2.0 ** -10))) == 0x80
    # 1.5 * 2^-9 halfway between codes 0x01 and 0x02 -> even 0x02
    assert oracle.e4m3_encode(np.float32(1.5 * 2.0 ** -9)) == 0x02
    # 1 + 1/16 halfway between 1.0 (0x38) and 1.125 (0x39) -> 0x38
    assert oracle.e4m3_encode(np.float32(1.0625)) == 0x38
    assert oracle.e4m3_encode(np.float32(-0.0)) == 0x80
    assert oracle.e4m3_encode(np.float32(449.0)) == 0x7E


@pytest.mark.parametrize("scale", [0.05, 1.0, 0.37, 3.0])
def test_quantize_is_fp32_division_then_rne(scale):
    x = _all_bf16_as_f32()
    x = x[np.isfinite(x)]
    sc = np.float32(scale)
    y = (torch.from_numpy(x.copy()) / torch.tensor(sc)).numpy()   # library fp32 division
    ok = np.abs(y) < 464.0
    ours = oracle.quantize_e4m3(x[ok], scale)
    ref = torch.from_numpy(y[ok].copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# -------------------------------------------------------------- slot / write

def test_worked_slot_example_write_and_walk():
    g = golden_kv("slot_worked_example.txt")
    B = int(g["block_size"][0])
    table = [int(v) for v in g["block_table"]]
    pos = int(g["position"][0])
    assert pos // B == int(g["logical_block"][0]) and pos % B == int(g["offset"][0])
    assert table[pos // B] == int(g["physical_block"][0])
    slot = int(g["slot"][0])
    # the write puts a row with slot 36 at flat row 36 = block 2, offset 4
    NB, Hkv, D = 16, 2, 8
    cache = np.zeros((NB * B, Hkv, D), dtype=np.float32)
    row = RNG.standard_normal((1, Hkv, D)).astype(np.float32)
    oracle.write_flat(row, "f32", np.array([slot]), cache, "f32")
    hnd = cache.reshape(NB, B, Hkv, D).transpose(0, 2, 1, 3)   # [block, head, offset, d]
    assert np.array_equal(hnd[slot // B, :, slot % B, :], row[0])
    assert np.count_nonzero(cache) == np.count_nonzero(row)
    # the paged walk reaches that row through the block table: give only it a large logit
    L = 3 * B
    q = np.ones((Hkv, D))
    pk = np.zeros((NB * B, Hkv, D))
    pv = np.zeros((NB * B, Hkv, D))
    pk[slot] = 10.0
    pv[slot] = row[0]
    out = oracle.paged_walk_decode(q, pk, pv, table, B, L, 1.0)
    assert np.allclose(out, row[0], atol=1e-12)


def test_debug_example_page_boundary():
    g = golden_kv("debug_example.txt")
    B = int(g["block_size"][0])
    table = [int(v) for v in g["block_table"]]
    t = int(g["logical_token"][0])
    L = int(g["seq_len"][0])
    assert (t // B, t % B, table[t // B]) == (int(g["logical_block"][0]), int(g["offset"][0]),
                                              int(g["physical_block"][0]))
    NB, Hkv, D = 16, 1, 4
    pk = np.zeros((NB * B, Hkv, D))
    pv = np.zeros((NB * B, Hkv, D))
    target = table[t // B] * B + t % B
    pk[target] = 50.0
    pv[target] = [1, 2, 3, 4]
    out = oracle.paged_walk_decode(np.ones((1, D)), pk, pv, table, B, L, 1.0)
    assert np.allclose(out[0], [1, 2, 3, 4], atol=1e-12)


def test_negative_slot_writes_nothing():
    T, Hkv, D, slots_n = 6, 3, 16, 64
    rows = RNG.standard_normal((T, Hkv, D)).astype(np.float32)
    rows[5] = np.nan
    slots = np.array([3, 17, -1, 40, 63, -1], dtype=np.int64)
    cache = np.full((slots_n, Hkv, D), 7.25, dtype=np.float32)
    before = cache.copy()
    oracle.write_flat(rows, "f32", slots, cache, "f32")
    written = {3: 0, 17: 1, 40: 3, 63: 4}
    for s in range(slots_n):
        if s in written:
            assert np.array_equal(cache[s], rows[written[s]])
        else:
            assert np.array_equal(cache[s].view(np.uint32), before[s].view(np.uint32))


def test_write_bf16_copies_bits_and_rejects_out_of_range():
    T, Hkv, D = 4, 2, 8
    bits = RNG.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
    cache = np.zeros((32, Hkv, D), dtype=np.uint16)
    oracle.write_flat(bits, "bf16", np.array([0, 5, 31, 7]), cache, "bf16")
    assert np.array_equal(cache[[0, 5, 31, 7]], bits)
    with pytest.raises(ValueError):
        oracle.write_flat(bits, "bf16", np.array([0, 5, 32, 7]), cache, "bf16")


def test_write_e4m3_quantises_each_element():
    T, Hkv, D = 3, 2, 16
    x = (RNG.standard_normal((T, Hkv, D)) * 3).astype(np.float32)
    bf = (x.view(np.uint32) >> 16).astype(np.uint16)           # truncated bf16 bit patterns
    vals = (bf.astype(np.uint32) << 16).view(np.float32)
    cache = np.zeros((8, Hkv, D), dtype=np.uint8)
    oracle.write_flat(bf, "bf16", np.array([2, -1, 6]), cache, "e4m3", 0.05)
    ref = torch.from_numpy((vals / np.float32(0.05)).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(cache[2], ref[0]) and np.array_equal(cache[6], ref[2])
    assert not cache[[0, 1, 3, 4, 5, 7]].any()


# ------------------------------------------------------------------- decode

def _rand(L, Hq, Hkv, D, rng=RNG):
    return rng.standard_normal((Hq, D)), rng.standard_normal((L, Hkv, D)), rng.standard_normal((L, Hkv, D))


def test_dense_mha_vs_scipy_softmax():
    for L, H, D in [(1, 1, 4), (7, 3, 16), (37, 4, 64), (200, 2, 128)]:
        q, K, V = _rand(L, H, H, D)
        scale = 1.0 / math.sqrt(D)
        out = oracle.dense_decode(q, K, V, scale)
        for h in range(H):
            p = softmax(scale * (K[:, h, :] @ q[h]))
            assert np.allclose(out[h], p @ V[:, h, :], rtol=1e-12, atol=1e-13)


def test_dense_gqa_vs_expanded_mha():
    L, Hq, Hkv, D = 50, 8, 2, 32
    q, K, V = _rand(L, Hq, Hkv, D)
    out = oracle.dense_decode(q, K, V, 0.3)
    Ke = np.repeat(K, Hq // Hkv, axis=1)   # query head h reads KV head h // (Hq/Hkv)
    Ve = np.repeat(V, Hq // Hkv, axis=1)
    for h in range(Hq):
        p = softmax(0.3 * (Ke[:, h, :] @ q[h]))
        assert np.allclose(out[h], p @ Ve[:, h, :], rtol=1e-12, atol=1e-13)


def test_gqa_head_map_golden():
    for Hq, Hkv, h, g in (map(int, r) for r in golden_lines("gqa_example.txt")):
        L, D = 3, 4
        q = RNG.standard_normal((Hq, D))
        K = RNG.standard_normal((L, Hkv, D))
        V = np.zeros((L, Hkv, D))
        for kv in range(Hkv):
            V[:, kv, :] = kv + 1.0        # output identifies the KV head read
        out = oracle.dense_decode(q, K, V, 1.0)
        assert np.allclose(out[h], g + 1.0, atol=1e-12)


def test_dense_closed_forms():
    D = 16
    # L = 1 -> o = v0
    q, K, V = _rand(1, 2, 2, D)
    assert np.array_equal(oracle.dense_decode(q, K, V, 0.25), V[0])
    # all keys equal -> mean of values
    q, K, V = _rand(9, 1, 1, D)
    K[:] = K[0]
    assert np.allclose(oracle.dense_decode(q, K, V, 0.25)[0], V[:, 0].mean(0), atol=1e-13)
    # q = 0 -> mean of values
    q[:] = 0
    K = RNG.standard_normal(K.shape)
    assert np.allclose(oracle.dense_decode(q, K, V, 0.25)[0], V[:, 0].mean(0), atol=1e-13)
    # two tokens: weight of token 0 is the logistic of the logit gap
    q, K, V = _rand(2, 1, 1, D)
    sc = 0.7
    z0, z1 = sc * K[0, 0] @ q[0], sc * K[1, 0] @ q[0]
    w0 = 1.0 / (1.0 + math.exp(z1 - z0))
    assert np.allclose(oracle.dense_decode(q, K, V, sc)[0], w0 * V[0, 0] + (1 - w0) * V[1, 0], atol=1e-13)
    # one logit 40 above the rest -> that token's value within e^-40
    L = 20
    q = np.zeros((1, D))
    q[0, 0] = 1.0
    K = np.zeros((L, 1, D))
    K[13, 0, 0] = 40.0
    V = RNG.standard_normal((L, 1, D))
    out = oracle.dense_decode(q, K, V, 1.0)
    assert np.allclose(out[0], V[13, 0], atol=L * math.exp(-40) * 10)
    # L = 0 -> zeros
    assert not oracle.dense_decode(np.ones((2, D)), np.zeros((0, 1, D)), np.zeros((0, 1, D)), 1.0).any()


def test_softmax_weights_sum_to_one_and_scale_equivariance():
    L, Hq, Hkv, D = 300, 4, 2, 64
    q, K, V = _rand(L, Hq, Hkv, D)
    out, p = oracle.dense_decode(q, K, V, 0.125, return_probs=True)
    assert np.all(p >= 0) and np.allclose(p.sum(1), 1.0, atol=1e-12)
    # scaling q by c and the softmax scale by 1/c changes nothing
    out2 = oracle.dense_decode(q * 4.0, K, V, 0.125 / 4.0)
    assert np.allclose(out, out2, rtol=1e-12, atol=1e-14)


def test_dense_token_permutation_invariance():
    L, Hq, Hkv, D = 64, 4, 4, 16
    q, K, V = _rand(L, Hq, Hkv, D)
    perm = RNG.permutation(L)
    a = oracle.dense_decode(q, K, V, 0.2)
    b = oracle.dense_decode(q, K[perm], V[perm], 0.2)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_paged_walk_equals_dense_under_block_permutations():
    B, Hq, Hkv, D = 16, 8, 2, 32
    rng = np.random.default_rng(99)
    for trial in range(24):
        L = int(rng.integers(1, 200))
        nb = (L + B - 1) // B
        NB = nb + int(rng.integers(0, 8))
        q, K, V = _rand(L, Hq, Hkv, D, rng)
        table = rng.permutation(NB)[:nb].astype(np.int32)
        pk = np.full((NB * B, Hkv, D), np.nan)      # unused slots poisoned
        pv = np.full((NB * B, Hkv, D), np.nan)
        for t in range(L):
            s = table[t // B] * B + t % B
            pk[s], pv[s] = K[t], V[t]
        a = oracle.dense_decode(q, K, V, 0.17)
        b = oracle.paged_walk_decode(q, pk, pv, table, B, L, 0.17)
        assert np.allclose(a, b, rtol=1e-12, atol=1e-13), trial
    # the out-of-order table [3, 1] from the pages' Python model
    L, NB = 8, 4
    Bs = 4
    q, K, V = _rand(L, 1, 1, 8, rng)
    pk = np.zeros((NB * Bs, 1, 8))
    pv = np.zeros((NB * Bs, 1, 8))
    table = [3, 1]
    for t in range(L):
        pk[table[t // Bs] * Bs + t % Bs] = K[t]
        pv[table[t // Bs] * Bs + t % Bs] = V[t]
    assert np.allclose(oracle.paged_walk_decode(q, pk, pv, table, Bs, L, 0.5),
                       oracle.dense_decode(q, K, V, 0.5), rtol=1e-12)


def test_partition_example_and_split_equals_unsplit():
    g = golden_kv("partition_example.txt")
    L, P, B = int(g["context_len"][0]), int(g["partition_size"][0]), int(g["block_size"][0])
    rows = [list(map(int, r)) for r in golden_lines("partition_example.txt") if r[0].isdigit()]
    nparts = -(-L // P)
    assert nparts == len(rows) == 3
    for p, first, last, nblocks, last_valid in rows:
        t0, t1 = p * P, min((p + 1) * P, L)
        assert (t0, t1 - 1) == (first, last)
        assert -(-(t1 - t0) // B) == nblocks
        assert (t1 - t0) - (nblocks - 1) * B == last_valid
    Hq, Hkv, D = 4, 2, 16
    q, K, V = _rand(L, Hq, Hkv, D)
    dense = oracle.dense_decode(q, K, V, 0.3)
    for P in (16, 48, 512, 2048):
        parts = [oracle.partial_decode(q, K, V, p * P, min((p + 1) * P, L), 0.3) for p in range(-(-L // P))]
        for h in range(Hq):
            m = np.array([pt[0][h] for pt in parts])
            l = np.array([pt[1][h] for pt in parts])
            acc = np.array([pt[2][h] for pt in parts])
            assert np.allclose(oracle.lse_merge(m, l, acc), dense[h], rtol=1e-12, atol=1e-13), (P, h)


def test_merge_identity_and_empty_parts():
    q, K, V = _rand(40, 2, 1, 8)
    m, l, acc = oracle.partial_decode(q, K, V, 0, 40, 1.0)
    one = oracle.lse_merge(m[:1], l[:1], acc[:1])
    assert np.allclose(one, acc[0] / l[0], rtol=1e-14)
    me, le, ae = oracle.partial_decode(q, K, V, 5, 5, 1.0)
    assert me[0] == -np.inf and le[0] == 0 and not ae.any()
    two = oracle.lse_merge(np.array([m[0], me[0]]), np.array([l[0], le[0]]), np.stack([acc[0], ae[0]]))
    assert np.allclose(two, one, rtol=1e-14)


def test_pool_constants_and_workload_sizes():
    g = golden_kv("pool_constants.txt")
    B, H, Dh, eb = (int(g[k][0]) for k in ("block_size", "kv_heads", "head_dim", "elem_bytes"))
    assert B * H * Dh * eb == int(g["v_offset_bytes"][0])
    assert 2 * int(g["v_offset_bytes"][0]) == int(g["block_bytes"][0])
    assert int(g["pool_bytes"][0]) // int(g["block_bytes"][0]) == int(g["num_blocks"][0])
    assert int(g["max_seq_len"][0]) // B == int(g["max_blocks_per_seq"][0])
    from workloads import configs
    w = configs.get("c2")
    assert w.num_blocks == int(g["num_blocks"][0]) and w.max_blocks == int(g["max_blocks_per_seq"][0])
    assert (w.Hkv, w.D) == (H, Dh)
    w1 = configs.get("c1")
    sw = golden_kv("slot_worked_example.txt")
    assert list(w1.block_table[1]) == [int(v) for v in sw["block_table"]]
    i = [k for k in range(w1.T) if w1.step_seq[k] == 1 and w1.step_pos[k] == int(sw["position"][0])][0]
    assert w1.step_slot[i] == int(sw["slot"][0])


@pytest.mark.parametrize("scale", [0.05, 0.37, 3.0])
def test_quantize_near_rounding_midpoints(scale):
    """fp32 inputs within a few ulps of (E4M3 midpoint) * scale: only a correctly
    rounded division followed by RNE matches the library conversion here (a
    multiply by the rounded reciprocal does not)."""
    mags = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2.0
    sc = np.float32(scale)
    base = (mids * float(sc)).astype(np.float32)
    xs = [base]
    for k in range(1, 4):
        xs.append(np.nextafter(xs[-1], np.float32(np.inf)))
    lo = [base]
    for k in range(1, 4):
        lo.append(np.nextafter(lo[-1], np.float32(0)))
    x = np.concatenate(xs + lo[1:])
    x = np.concatenate([x, -x])
    y = (torch.from_numpy(x.copy()) / torch.tensor(sc)).numpy()
    ok = np.abs(y) < 464.0
    ref = torch.from_numpy(y[ok].copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.quantize_e4m3(x[ok], scale), ref)


# ------------------------------------------ per-head scales, ALiBi, multi-query

def test_write_per_head_scales():
    """Head h quantises with its own scale ("Inside vLLM CUDA Kernels", Part 2: head h uses
    scale[h * kv_scale_stride]): each head against the library's fp32 division and E4M3
    conversion with that head's scale; equal per-head scales give the per-tensor write."""
    T, Hkv, D = 5, 4, 16
    x = (RNG.standard_normal((T, Hkv, D)) * 3).astype(np.float32)
    bf = (x.view(np.uint32) >> 16).astype(np.uint16)
    vals = (bf.astype(np.uint32) << 16).view(np.float32)
    scales = np.array([0.05, 0.37, 1.0, 3.0], dtype=np.float32)
    slots = np.array([3, -1, 0, 7, 5])
    cache = np.zeros((8, Hkv, D), dtype=np.uint8)
    oracle.write_flat(bf, "bf16", slots, cache, "e4m3", scales)
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        for h in range(Hkv):
            y = (torch.from_numpy(vals[t, h].copy()) / torch.tensor(scales[h])).numpy()
            assert np.abs(y).max() < 464.0
            ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(cache[sl, h], ref), (t, h)
    assert not cache[[1, 2, 4, 6]].any()
    same, per_tensor = np.zeros_like(cache), np.zeros_like(cache)
    oracle.write_flat(bf, "bf16", slots, same, "e4m3", np.full(Hkv, 0.37, np.float32))
    oracle.write_flat(bf, "bf16", slots, per_tensor, "e4m3", 0.37)
    assert np.array_equal(same, per_tensor)
    # element values with per-head scales: the library's E4M3 decode times the head's scale
    v = oracle.cache_values(cache, "e4m3", scales)
    lib_vals = torch.from_numpy(cache.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(v, lib_vals * scales.astype(np.float64)[None, :, None])


def test_alibi_closed_form():
    """q = 0 makes every dot product 0, so the weights are exp(a (t - (L - 1))) normalised: a
    geometric distribution with ratio e^-a, ending at the current position (bias 0).  With
    V[t] = e_t the output is that distribution."""
    L, D = 12, 16
    for a in (0.0, 0.25, 1.5, 40.0):
        q = np.zeros((1, 1, D))
        K = RNG.standard_normal((L, 1, D))
        V = np.zeros((L, 1, D))
        V[np.arange(L), 0, np.arange(L)] = 1.0
        out = oracle.attention_causal(q, K, V, 0.7, alibi_slopes=[a])[0, 0]
        r = math.exp(-a)
        ref = np.array([r ** (L - 1 - t) for t in range(L)])
        ref /= ref.sum()
        assert np.allclose(out[:L], ref, rtol=1e-12, atol=1e-300) and not out[L:].any()


def test_alibi_decode_vs_scipy_softmax_and_zero_slopes():
    L, Hq, Hkv, D = 40, 4, 2, 16
    q, K, V = _rand(L, Hq, Hkv, D)
    slopes = np.array([0.5, 0.0625, 2.0 ** -8, 1.0])
    out = oracle.attention_causal(q[None], K, V, 0.25, slopes)[0]
    G = Hq // Hkv
    for h in range(Hq):
        z = 0.25 * (K[:, h // G, :] @ q[h]) + slopes[h] * (np.arange(L) - (L - 1))
        assert np.allclose(out[h], softmax(z) @ V[:, h // G, :], rtol=1e-12, atol=1e-13)
    # zero slopes (or none): single-query decode
    assert np.array_equal(oracle.attention_causal(q[None], K, V, 0.25, np.zeros(Hq))[0],
                          oracle.attention_causal(q[None], K, V, 0.25)[0])
    assert np.allclose(oracle.attention_causal(q[None], K, V, 0.25)[0], oracle.dense_decode(q, K, V, 0.25),
                       rtol=1e-13, atol=1e-14)


def test_causal_whole_prompt_vs_masked_matrix():
    """n = L (a whole prompt): the textbook masked form softmax(scale Q K^T + bias + M) V, M the
    strictly-upper-triangular -inf mask, bias a_h (j - i)."""
    L, Hq, Hkv, D = 9, 4, 2, 8
    q = RNG.standard_normal((L, Hq, D))
    K = RNG.standard_normal((L, Hkv, D))
    V = RNG.standard_normal((L, Hkv, D))
    slopes = np.array([0.0, 0.5, 0.125, 2.0])
    out = oracle.attention_causal(q, K, V, 0.3, slopes)
    G = Hq // Hkv
    idx = np.arange(L)
    for h in range(Hq):
        Z = 0.3 * q[:, h, :] @ K[:, h // G, :].T + slopes[h] * (idx[None, :] - idx[:, None])
        Z[np.triu_indices(L, 1)] = -np.inf
        assert np.allclose(out[:, h, :], softmax(Z, axis=1) @ V[:, h // G, :], rtol=1e-12, atol=1e-13)


def test_causal_chunk_rows_are_prefix_decodes():
    """n < L (new tokens at the end of a history): query i is single-query decode over the
    first L - n + i + 1 tokens; more queries than history is refused."""
    L, n, Hq, Hkv, D = 30, 5, 8, 2, 16
    q = RNG.standard_normal((n, Hq, D))
    K = RNG.standard_normal((L, Hkv, D))
    V = RNG.standard_normal((L, Hkv, D))
    out = oracle.attention_causal(q, K, V, 0.2)
    for i in range(n):
        vis = L - n + i + 1
        assert np.allclose(out[i], oracle.dense_decode(q[i], K[:vis], V[:vis], 0.2), rtol=1e-13, atol=1e-14)
    with pytest.raises(ValueError):
        oracle.attention_causal(np.zeros((4, 2, 8)), np.zeros((3, 1, 8)), np.zeros((3, 1, 8)), 1.0)
