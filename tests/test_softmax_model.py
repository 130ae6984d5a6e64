"""The numerical recipe of the tensor-core attention kernels, modelled on the CPU in
float32 with 16-bit rounding where the kernels round, against the fp64 oracle.

Both kernels (the decode kernel per 16-token page, the query-tile kernel per 64-token
group) keep, per query column, a running max m in log2 units that moves only when a
score exceeds it by more than 8, weights p = 2^(s - m) (so p <= 256), a float32 row sum
and a float32 output accumulator, and feed P to the tensor cores as two 16-bit halves
(hi = RN16(p), lo = RN16(p - hi)) against 16-bit V.  The model checks that recipe meets
the parity bar |out - oracle| <= 1e-3 + 1 bf16 ulp on ordinary and adversarial score
patterns, and that P in one 16-bit half does not (the reason the kernels pay for the
second P.V product)."""
import math
import zlib

import numpy as np
import pytest

import oracle

SLACK = 8.0


def rn_bf16(x):
    """float32 -> bfloat16 (round to nearest even) -> float32."""
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def model(q, K, V, scale, group, split_p=True):
    """One query row: q [D] (already bf16 values), K, V [L, D] (bf16 values)."""
    q32, K32, V32 = q.astype(np.float32), K.astype(np.float32), V.astype(np.float32)
    sl2 = np.float32(scale * math.log2(math.e))
    m, l = np.float32(-1e30), np.float32(0.0)
    acc = np.zeros(q.shape[0], dtype=np.float32)
    for t0 in range(0, K.shape[0], group):
        s = (K32[t0:t0 + group] @ q32).astype(np.float32) * sl2
        lm = np.float32(s.max())
        if lm > m + SLACK:
            alpha = np.float32(2.0) ** (m - lm)
            l *= alpha
            acc *= alpha
            m = lm
        p = (np.float32(2.0) ** (s - m)).astype(np.float32)
        l += np.float32(p.sum(dtype=np.float32))
        hi = rn_bf16(p)
        lo = rn_bf16(p - hi) if split_p else np.zeros_like(p)
        acc += (hi @ V32[t0:t0 + group]).astype(np.float32) + (lo @ V32[t0:t0 + group]).astype(np.float32)
    return acc / l


def bar(got, ref):
    ulp = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(ref), 1e-38))), -126) - 7)
    return np.abs(got - ref) <= 1e-3 + ulp


def case(kind, L, D, rng):
    q = rn_bf16(rng.standard_normal(D))
    K = rn_bf16(rng.standard_normal((L, D)))
    V = rn_bf16(rng.standard_normal((L, D)))
    scale = 1.0 / math.sqrt(D)
    if kind == "outlier":      # one key +20 above the rest (the long-context workload's pattern)
        t = int(rng.integers(L))
        K[t] = rn_bf16(q * (20.0 / (scale * float(q @ q))))
    elif kind == "rising":     # scores growing along the sequence: the running max moves often
        K = rn_bf16(K * 0.2 + np.outer(np.linspace(0, 6, L), q) / math.sqrt(float(q @ q)))
    elif kind == "two_opposed":  # two dominant keys (logits 25 and 24.7) whose values cancel
        a, b = rng.choice(L, size=2, replace=False)
        K[a] = rn_bf16(q * (25.0 / (scale * float(q @ q))))
        K[b] = rn_bf16(q * (24.7 / (scale * float(q @ q))))
        za, zb = scale * float(K[a] @ q), scale * float(K[b] @ q)
        V[a] = rn_bf16(V[a] * 3.0)
        V[b] = rn_bf16(-V[a] * math.exp(za - zb) * 0.999)
    return q, K, V, scale


@pytest.mark.parametrize("kind", ["random", "outlier", "rising", "two_opposed"])
@pytest.mark.parametrize("group", [16, 64])
def test_recipe_meets_the_parity_bar(kind, group):
    rng = np.random.default_rng(zlib.crc32(("%s/%d" % (kind, group)).encode()))
    for L, D in ((1, 64), (17, 64), (300, 128), (2000, 128)):
        if kind == "two_opposed" and L < 2:
            continue
        q, K, V, scale = case(kind, L, D, rng)
        ref = oracle.dense_decode(q.astype(np.float64)[None], K.astype(np.float64)[:, None],
                                  V.astype(np.float64)[:, None], scale)[0]
        got = model(q, K, V, scale, group)
        assert bar(got, ref).all(), (kind, group, L, D, float(np.abs(got - ref).max()))


def test_one_half_of_p_misses_the_bar():
    """Negative control: with P rounded to one bf16 half, a row whose output is a small
    difference of large contributions misses the bar somewhere in a batch of such rows."""
    rng = np.random.default_rng(5)
    misses = 0
    for _ in range(40):
        q, K, V, scale = case("two_opposed", 64, 128, rng)
        ref = oracle.dense_decode(q.astype(np.float64)[None], K.astype(np.float64)[:, None],
                                  V.astype(np.float64)[:, None], scale)[0]
        full = model(q, K, V, scale, 16)
        half = model(q, K, V, scale, 16, split_p=False)
        assert bar(full, ref).all()
        misses += int((~bar(half, ref)).any())
    assert misses > 0
