"""The C-ABI library: it loads without a GPU, exports every function include/pa.h
declares, and its host-only logic (argument validation, partition plan, workspace
size) behaves as documented.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

from conftest import ROOT, golden_kv

import paged_decode_attention_reshape_gb300 as pa
from paged_decode_attention_reshape_gb300 import PaTensor


@pytest.fixture(scope="module")
def L():
    from paged_decode_attention_reshape_gb300 import _build
    _build.build()
    return pa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(pa.EXPORTS)


def test_status_strings(L):
    for code in range(0, -9, -1):
        s = pa.pa_status_string(code)
        assert s and s != "unknown status"
    assert pa.pa_status_string(-99) == "unknown status"


def _t(shape, dtype, ptr=0x10000, strides=None):
    d = PaTensor()
    d.data = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    if strides is None:
        strides = []
        acc = 1
        for n in reversed(shape):
            strides.insert(0, acc)
            acc *= n
    for i, (n, s) in enumerate(zip(shape, strides)):
        d.shape[i] = n
        d.stride[i] = s
    return d


def _write(L, key, value, kc, vc, sm, mode=pa.PA_KV_AUTO):
    return L.pa_reshape_and_cache(ctypes.byref(key), ctypes.byref(value), ctypes.byref(kc), ctypes.byref(vc),
                                  ctypes.byref(sm), mode, None, None, None, None)


def test_write_validation(L):
    T, H, D, NB = 4, 2, 64, 8
    key = _t([T, H, D], pa.PA_BF16)
    val = _t([T, H, D], pa.PA_BF16)
    kc = _t([NB, H, 16, D], pa.PA_BF16)
    vc = _t([NB, H, 16, D], pa.PA_BF16)
    sm = _t([T], pa.PA_I64)
    # T == 0 is a no-op that returns before touching the device
    assert _write(L, _t([0, H, D], pa.PA_BF16), _t([0, H, D], pa.PA_BF16), kc, vc, _t([0], pa.PA_I64)) == 0
    assert _write(L, key, val, kc, vc, _t([T], pa.PA_I32)) == -2                  # slot_mapping not int64
    assert _write(L, key, _t([T, H, D], pa.PA_F16), kc, vc, sm) == -1            # key/value types differ
    assert _write(L, key, val, _t([NB, H, 8, D], pa.PA_BF16), _t([NB, H, 8, D], pa.PA_BF16), sm) == -7  # block 8
    assert _write(L, key, val, _t([NB, H, 16, D], pa.PA_F16), _t([NB, H, 16, D], pa.PA_F16), sm) == -2
    assert _write(L, key, val, kc, vc, sm, pa.PA_KV_FP8_E4M3) == -2              # fp8 mode, bf16 cache
    assert _write(L, key, val, kc, vc, sm, 7) == -1                              # unknown mode
    assert _write(L, _t([T, H + 1, D], pa.PA_BF16), _t([T, H + 1, D], pa.PA_BF16), kc, vc, sm) == -1
    assert _write(L, key, val, kc, vc, _t([T + 1], pa.PA_I64)) == -1
    assert _write(L, key, val, _t([NB, H, 16, D], pa.PA_BF16, ptr=0x10008), vc, sm) == -3  # misaligned cache
    assert _write(L, _t([T, H, D], pa.PA_BF16, ptr=0x10004), val, kc, vc, sm) == -3        # misaligned key
    assert _write(L, key, val, kc, vc, _t([T], pa.PA_I64, ptr=0)) == -1           # null slot_mapping
    bad = _t([T, H, D], pa.PA_BF16, strides=[H * D, D, 2])                        # inner stride != 1
    assert _write(L, bad, val, kc, vc, sm) == -1


def _decode(L, out, q, kc, vc, bt, sl, hkv, psize=0, ws=None, ws_bytes=0):
    return L.pa_decode_ex(ctypes.byref(out), ctypes.byref(q), ctypes.byref(kc), ctypes.byref(vc), ctypes.byref(bt),
                          ctypes.byref(sl), 0.125, hkv, None, None, psize, ws, ws_bytes, None, None)


def test_decode_validation(L):
    S, Hq, Hkv, D, NB, MB = 3, 8, 2, 128, 16, 4
    q = _t([S, Hq, D], pa.PA_BF16)
    out = _t([S, Hq, D], pa.PA_BF16, ptr=0x20000)
    kc = _t([NB, Hkv, 16, D], pa.PA_BF16)
    vc = _t([NB, Hkv, 16, D], pa.PA_BF16)
    bt = _t([S, MB], pa.PA_I32)
    sl = _t([S], pa.PA_I32)
    assert _decode(L, _t([0, Hq, D], pa.PA_BF16), _t([0, Hq, D], pa.PA_BF16), kc, vc, _t([0, MB], pa.PA_I32),
                   _t([0], pa.PA_I32), Hkv) == 0                                  # empty batch: no-op
    assert _decode(L, out, q, kc, vc, bt, sl, 3) == -1                           # num_kv_heads mismatch
    assert _decode(L, out, _t([S, 7, D], pa.PA_BF16), kc, vc, bt, sl, Hkv) == -1  # out/q shapes differ
    assert _decode(L, _t([S, Hq, D], pa.PA_F16), q, kc, vc, bt, sl, Hkv) == -1   # out dtype != q dtype
    assert _decode(L, out, q, kc, vc, _t([S, MB], pa.PA_I64), sl, Hkv) == -2     # table not int32
    assert _decode(L, out, q, kc, vc, bt, _t([S + 1], pa.PA_I32), Hkv) == -1
    kf = _t([NB, Hkv, 16, D], pa.PA_F16)
    assert _decode(L, out, q, kf, _t([NB, Hkv, 16, D], pa.PA_F16), bt, sl, Hkv) == -2   # bf16 q, f16 cache
    k8 = _t([NB, Hkv, 16, 64], pa.PA_FP8_E4M3)
    assert _decode(L, _t([S, Hq, 64], pa.PA_BF16), _t([S, Hq, 64], pa.PA_BF16), k8,
                   _t([NB, Hkv, 16, 64], pa.PA_FP8_E4M3), bt, sl, Hkv) == -7     # fp8 needs D >= 128
    k96 = _t([NB, Hkv, 16, 96], pa.PA_BF16)
    assert _decode(L, _t([S, Hq, 96], pa.PA_BF16), _t([S, Hq, 96], pa.PA_BF16), k96,
                   _t([NB, Hkv, 16, 96], pa.PA_BF16), bt, sl, Hkv) == -7         # head size not built
    assert _decode(L, out, _t([S, Hq, D], pa.PA_BF16, ptr=0x10002), kc, vc, bt, sl, Hkv) == -3
    assert _decode(L, out, q, kc, _t([NB, Hkv, 16, D], pa.PA_BF16, strides=[Hkv * 16 * D, 16 * D, D + 4, 1]),
                   bt, sl, Hkv) == -3                                            # token stride not 16 B
    assert _decode(L, out, q, kc, _t([NB + 1, Hkv, 16, D], pa.PA_BF16), bt, sl, Hkv) == -1  # K/V extents differ
    assert _decode(L, out, q, _t([NB, Hkv, 16, D], pa.PA_BF16, strides=[Hkv * 16 * D + 4, 16 * D, D, 1]),
                   vc, bt, sl, Hkv) == -3                                        # block stride not 16 B


def test_partition_plan_golden_example(L):
    """The 1100-token example at 512-token partitions: 3 partitions."""
    g = golden_kv("partition_example.txt")
    ctx, P = int(g["context_len"][0]), int(g["partition_size"][0])
    max_blocks = -(-ctx // 16)
    part, n = pa.pa_decode_plan(1, 8, 2, 128, max_blocks, pa.PA_BF16, 152, P)
    assert part == 512 and n == 3


def test_partition_plan_rules(L):
    # -1 never splits; explicit sizes round up to whole pages; a partition covering the longest
    # possible sequence is no split at all
    assert pa.pa_decode_plan(4, 32, 8, 128, 8192, pa.PA_BF16, 152, -1) == (0, 1)
    assert pa.pa_decode_plan(4, 32, 8, 128, 8192, pa.PA_BF16, 152, 500) == (512, 256)
    assert pa.pa_decode_plan(4, 32, 8, 128, 8, pa.PA_BF16, 152, 512) == (0, 1)
    # -2 / -4 / -8: cluster split into that many equal parts; other negative values are invalid
    for C in (2, 4, 8):
        assert pa.pa_decode_plan(4, 32, 8, 128, 8192, pa.PA_BF16, 152, -C) == (-C, C)
    for bad in (-3, -5, -16):
        with pytest.raises(pa.PAError):
            pa.pa_decode_plan(4, 32, 8, 128, 8192, pa.PA_BF16, 152, bad)
    # heuristic: a few long sequences get fixed partitions, never below 1024 tokens
    P, n = pa.pa_decode_plan(4, 32, 8, 128, 8192, pa.PA_BF16, 152, 0)
    assert P >= 1024 and P % 16 == 0 and n == -(-8192 * 16 // P) and n > 8
    # heuristic: a batch that fits the resident slots gets its longest sequences cut in two
    assert pa.pa_decode_plan(64, 32, 8, 128, 128, pa.PA_BF16, 300, 0) == (1024, 2)
    # heuristic: a longest-first batch whose units fill the slots once (64 x 8 units, 152 x 3
    # resident 8-warp CTAs at head size 64) is not split
    assert pa.pa_decode_plan(64, 32, 8, 64, 128, pa.PA_BF16, 152, 0) == (0, 1)
    # heuristic: a partition as long as the table is no split
    assert pa.pa_decode_plan(64, 32, 8, 64, 64, pa.PA_BF16, 152, 0) == (0, 1)
    # heuristic: a longest-first batch whose units fill the resident slots is not split
    assert pa.pa_decode_plan(128, 64, 8, 128, 512, pa.PA_FP8_E4M3, 152, 0) == (0, 1)
    # heuristic: many (sequence, kv head) units fill the GPU without splitting
    assert pa.pa_decode_plan(4096, 32, 8, 128, 256, pa.PA_BF16, 152, 0) == (0, 1)
    # invalid arguments
    with pytest.raises(pa.PAError):
        pa.pa_decode_plan(4, 30, 8, 128, 64, pa.PA_BF16, 152, 0)


def test_balanced_split_plan(L):
    """PA_PARTITION_BALANCED: one resident wave of CTAs per (kv head, head group) row.
    Without a device the resident CTAs per SM are the shared-memory bound:
    D=64 bf16 pages 2 KiB -> 8 warps x 2 stages x 4 KiB + 3 KiB = 67 KiB -> 3 per SM;
    D=128 bf16 -> 4 warps x 2 stages x 8 KiB + 3 KiB = 67 KiB -> 3 per SM."""
    B = pa.PA_PARTITION_BALANCED
    assert pa.pa_decode_plan(64, 32, 8, 64, 128, pa.PA_BF16, 152, B) == (B, 152 * 3 // 8)
    assert pa.pa_decode_plan(4, 32, 8, 128, 8192, pa.PA_BF16, 152, B) == (B, 152 * 3 // 8)
    assert pa.pa_decode_plan(4, 32, 2, 128, 8192, pa.PA_BF16, 152, B) == (B, 152 * 3 // 4)   # 2 groups per KV head
    assert pa.pa_decode_plan(1, 1024, 1024, 128, 8, pa.PA_BF16, 10, B) == (B, 1)              # fewer slots than rows
    assert pa.pa_decode_plan(511, 32, 8, 64, 128, pa.PA_BF16, 152, B)[0] == B
    with pytest.raises(pa.PAError) as e:                                                      # batch limit
        pa.pa_decode_plan(512, 32, 8, 64, 128, pa.PA_BF16, 152, B)
    assert e.value.status == -7
    assert pa.pa_decode_plan(4, 32, 8, 128, 64, pa.PA_F32, 152, B) == (0, 1)                 # fp32 kernel: unsplit


def test_workspace_size(L):
    S, Hq, Hkv, D, MB = 4, 32, 8, 128, 8192
    assert pa.pa_decode_workspace_size(S, Hq, Hkv, D, MB, 0) == 0
    assert pa.pa_decode_workspace_size(S, Hq, Hkv, D, MB, -1) == 0
    assert pa.pa_decode_workspace_size(S, Hq, Hkv, D, MB, -4) == 0           # cluster split: no workspace
    assert pa.pa_decode_workspace_size(S, 30, Hkv, D, MB, 512) == 0           # Hq % Hkv != 0
    parts = -(-MB * 16 // 512)
    rows = S * Hq * parts
    r256 = lambda x: (x + 255) // 256 * 256
    counters = r256(S * Hkv * 1 * 4)                                           # one per (seq, kv head, 8-head group)
    assert pa.pa_decode_workspace_size(S, Hq, Hkv, D, MB, 512) == counters + r256(rows * 8) + rows * D * 4
    # 16 query heads per KV head -> two head groups per KV head
    counters2 = r256(S * 2 * 2 * 4)
    rows2 = S * 32 * parts
    assert pa.pa_decode_workspace_size(S, 32, 2, D, MB, 512) == counters2 + r256(rows2 * 8) + rows2 * D * 4


def test_check_device_error_rejects_null(L):
    assert L.pa_check_device_error(None, None, None) == -1


def test_option_struct_layouts_match_the_header(tmp_path):
    """The binding's ctypes structs have the C header's size and field offsets."""
    import subprocess
    src = tmp_path / "offsets.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "pa.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\n", sizeof(pa_write_options), offsetof(pa_write_options, k_scale),
         offsetof(pa_write_options, v_scale), offsetof(pa_write_options, scale_stride),
         offsetof(pa_write_options, device_error));
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(pa_decode_options), offsetof(pa_decode_options, k_scale),
         offsetof(pa_decode_options, v_scale), offsetof(pa_decode_options, scale_stride),
         offsetof(pa_decode_options, alibi_slopes), offsetof(pa_decode_options, partition_size),
         offsetof(pa_decode_options, workspace), offsetof(pa_decode_options, workspace_bytes),
         offsetof(pa_decode_options, device_error));
  return 0;
}
''')
    exe = tmp_path / "offsets"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.check_call(["gcc", "-I", inc, "-o", str(exe), str(src)])
    w, d = [list(map(int, l.split())) for l in subprocess.check_output([str(exe)]).decode().split("\n")[:2]]
    W, D = pa.PaWriteOptions, pa.PaDecodeOptions
    assert w == [ctypes.sizeof(W)] + [getattr(W, f).offset for f in ("k_scale", "v_scale", "scale_stride",
                                                                      "device_error")]
    assert d == [ctypes.sizeof(D)] + [getattr(D, f).offset for f in ("k_scale", "v_scale", "scale_stride",
                                                                      "alibi_slopes", "partition_size", "workspace",
                                                                      "workspace_bytes", "device_error")]


def test_negative_scale_stride_is_refused(L):
    o = pa.PaDecodeOptions()
    o.scale_stride = -1
    assert L.pa_decode_opt(None, None, None, None, None, None, 1.0, 1, ctypes.byref(o), None) == -1
    w = pa.PaWriteOptions()
    w.scale_stride = -2
    assert L.pa_reshape_and_cache_opt(None, None, None, None, None, 0, ctypes.byref(w), None) == -1


def _step(L, out, q, key, val, kc, vc, sm, nrs, bt, sl, hkv):
    return L.pa_decode_step(ctypes.byref(out), ctypes.byref(q), ctypes.byref(key), ctypes.byref(val),
                            ctypes.byref(kc), ctypes.byref(vc), ctypes.byref(sm),
                            None if nrs is None else ctypes.byref(nrs), ctypes.byref(bt), ctypes.byref(sl), 0.125,
                            hkv, None, None)


def test_step_validation(L):
    """pa_decode_step checks the decode's arguments and the row mapping before it launches
    anything (the write's own checks come next, still before its launch)."""
    S, Hq, Hkv, D, NB, MB = 3, 8, 2, 128, 16, 4
    q = _t([S, Hq, D], pa.PA_BF16)
    out = _t([S, Hq, D], pa.PA_BF16, ptr=0x20000)
    kc = _t([NB, Hkv, 16, D], pa.PA_BF16)
    vc = _t([NB, Hkv, 16, D], pa.PA_BF16)
    bt = _t([S, MB], pa.PA_I32)
    sl = _t([S], pa.PA_I32)
    key = _t([S, Hkv, D], pa.PA_BF16)
    val = _t([S, Hkv, D], pa.PA_BF16)
    sm = _t([S], pa.PA_I64)
    # one row per sequence unless new_rows_start says otherwise
    assert _step(L, out, q, _t([S + 1, Hkv, D], pa.PA_BF16), _t([S + 1, Hkv, D], pa.PA_BF16), kc, vc,
                 _t([S + 1], pa.PA_I64), None, bt, sl, Hkv) == -1
    assert _step(L, out, q, key, val, kc, vc, sm, _t([S], pa.PA_I32), bt, sl, Hkv) == -1      # needs S + 1
    assert _step(L, out, q, key, val, kc, vc, sm, _t([S + 1], pa.PA_I64), bt, sl, Hkv) == -2  # int32 only
    assert _step(L, out, q, key, val, kc, vc, sm, None, bt, sl, 3) == -1                      # decode side
    assert _step(L, out, _t([S, 7, D], pa.PA_BF16), key, val, kc, vc, sm, None, bt, sl, Hkv) == -1
