#!/usr/bin/env python3
"""Benchmark of the paged KV-cache hot path on GB300.

One step = one pass of the whole path over one batch: the cache write of the
step's new tokens followed by paged decode attention (pa_decode_step: the write,
then the decode kernel with its fused split-KV merge when the plan splits).

Headline workload (``--config``, default c3): the 8B-class batched decode (256
sequences, 32 query / 8 KV heads, head size 128, bf16, lengths uniform in
[512, 4096], 256 new tokens written per step) -- the largest configuration.  The
same line carries, under ``configs``, the same measurement of the other
workloads (c2 small GQA decode, c4 long-context split-KV decode, c5 FP8 write +
decode, c3-chunk128 chunked prefill on the query-tile kernel).  L2 is flushed (a
512 MiB write and a 512 MiB read) before every timed step, outside the events.

Per workload: ``value`` = paged-decode KV-read GB/s over the whole step
(algorithmic decode bytes / step time; the step is captured once in a CUDA graph
and replayed, as a serving loop replays its decode step; ``eager_ms_per_step``
times the calls issued one by one from Python); ``roofline`` is for the attention
kernel alone (profiling events on its launch stream); ``e2e`` repeats the step
from pinned host buffers with the host<->device copies inside the timed region;
``cpu_baseline`` times the fp64 CPU oracle on a bounded sample of the same
workload.  ``--impl reference`` times that oracle as the reference arm;
``--sweep-partitions`` times the decode kernel over the partition sizes the
library's partition plan is fitted to.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import configs, data  # noqa: E402

METRIC = "paged-decode KV-read GB/s (% of HBM peak), tokens/s; cache-write GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Evict the L2 between timed steps: write a 512 MiB buffer (4x the 129 MB L2), then read
    another one, so the written lines are cleaned out too and the next timed kernel does not
    pay for their write-back."""

    def __init__(self, device):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()
DECODE_SOURCES = ["pa_decode_mma.cuh", "pa_decode_mma16.cu", "pa_decode_mma_fp8.cu", "pa_decode.cu",
                  "pa_device.cuh", "pa_internal.h", "pa_merge.cuh", "pa_api.cu"]
# sources of the query-tile kernel (chunked prefill / long query chunks)
CHUNK_SOURCES = ["pa_chunk_umma.cuh", "pa_chunk_mma16.cu", "pa_device.cuh", "pa_internal.h", "pa_api.cu"]


# ----------------------------------------------------------------- staging

class Staged:
    """Device-resident inputs and outputs of one workload."""


def _torch_dt(name):
    return {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}[name]


def nan_fill_(t: torch.Tensor) -> None:
    """Poison a cache with NaN bit patterns (all bytes 0xFF is NaN for fp32, bf16, f16, e4m3)."""
    t.view(torch.uint8).fill_(0xFF)


def stage(w, device="cuda", history=True, poison=True) -> Staged:
    """Allocate the cache pool (NaN-poisoned), write the history rows through the library's own
    cache write, and stage this step's new rows, metadata and output buffers on `device`."""
    import paged_decode_attention_reshape_gb300 as pa
    st = Staged()
    st.w = w
    cdt = _torch_dt(w.cache_dtype)
    nhd = w.layout == "nhd"
    shape = (w.num_blocks, configs.BLOCK, w.Hkv, w.D) if nhd else (w.num_blocks, w.Hkv, configs.BLOCK, w.D)
    kb = torch.empty(shape, dtype=cdt, device=device)
    vb = torch.empty(shape, dtype=cdt, device=device)
    if poison:
        nan_fill_(kb)
        nan_fill_(vb)
    # the library takes every cache as [NB, Hkv, 16, D]; an NHD cache is passed as that permutation
    st.k_cache = kb.permute(0, 2, 1, 3) if nhd else kb
    st.v_cache = vb.permute(0, 2, 1, 3) if nhd else vb
    st.fp8 = w.kv_dtype == "e4m3"
    st.kv_mode = pa.PA_KV_FP8_E4M3 if st.fp8 else pa.PA_KV_AUTO
    st.k_scale = torch.tensor(np.atleast_1d(w.k_scales()), dtype=torch.float32, device=device)
    st.v_scale = torch.tensor(np.atleast_1d(w.v_scales()), dtype=torch.float32, device=device)
    st.scale_stride = 0 if w.k_head_scales is None else 1
    st.alibi = None if w.alibi is None else torch.from_numpy(w.alibi).to(device)
    st.err = torch.zeros(1, dtype=torch.int32, device=device)
    bt = w.block_table.copy()
    st.block_table = torch.from_numpy(bt).to(device)
    st.seq_lens = torch.from_numpy(w.seq_lens.astype(np.int32)).to(device)
    st.q = data.q(w, device)
    st.out = torch.empty_like(st.q)
    # several query tokens per sequence: sequence s owns q / out rows s * nq .. s * nq + nq - 1
    st.qsl = torch.arange(0, w.S * w.nq + 1, w.nq, dtype=torch.int32, device=device) if w.nq > 1 else None
    st.k_step, st.v_step = data.step_rows(w, device)
    st.slot_mapping = torch.from_numpy(w.step_slot.astype(np.int64)).to(device)
    st.new_rows_start = new_rows_start(w, device)
    if history:
        write_history(st, device)
    return st


def new_rows_start(w, device="cuda"):
    """How the step's rows map to sequences for pa_decode_step: None when row s is sequence
    s's newest token, an int32 [S+1] tensor when each sequence's rows are its newest tokens in
    order, sequence after sequence (c5's chunk), and False when the step's rows are not its
    sequences' newest tokens (then the write and the attention are two calls)."""
    if w.nq != 1:
        return False
    seqs, pos = np.asarray(w.step_seq), np.asarray(w.step_pos)
    if len(seqs) == w.S and np.array_equal(seqs, np.arange(w.S)) and np.array_equal(pos, w.seq_lens - 1):
        return None
    if len(seqs) == 0 or seqs.min() < 0:   # a row of no sequence (padding tagged -1)
        return False
    counts = np.bincount(seqs, minlength=w.S)
    start = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    if not np.all(np.diff(seqs) >= 0):
        return False
    for s in range(w.S):
        n = int(counts[s])
        if not np.array_equal(pos[start[s]:start[s + 1]], np.arange(int(w.seq_lens[s]) - n, int(w.seq_lens[s]))):
            return False
    return torch.from_numpy(start).to(device)


def write_history(st: Staged, device="cuda", rows_per_call=1 << 16) -> None:
    """Every position [0, L_s) of every sequence gets its history row (the step overwrites some)."""
    import paged_decode_attention_reshape_gb300 as pa
    w = st.w
    for s in range(w.S):
        L = int(w.seq_lens[s])
        for p0 in range(0, L, rows_per_call):
            p1 = min(L, p0 + rows_per_call)
            pos = torch.arange(p0, p1, dtype=torch.int64)
            K, V = data.history_rows(w, s, device, positions=pos)
            slots = torch.from_numpy(w.slot_of(s, np.arange(p0, p1))).to(device)
            write_rows(st, K, V, slots)
    torch.cuda.synchronize()


def write_rows(st: Staged, K, V, slots) -> None:
    """Cache write of rows K/V [n, Hkv, D] at `slots` (the plain entry point unless the
    workload has per-head scales)."""
    import paged_decode_attention_reshape_gb300 as pa
    if st.scale_stride:
        pa.pa_reshape_and_cache_opt(K, V, st.k_cache, st.v_cache, slots, st.kv_mode, st.k_scale, st.v_scale,
                                    st.scale_stride, st.err)
    else:
        pa.pa_reshape_and_cache(K, V, st.k_cache, st.v_cache, slots, st.kv_mode, st.k_scale, st.v_scale, st.err)


def workspace_for(st: Staged, partition_size: int):
    import paged_decode_attention_reshape_gb300 as pa
    w = st.w
    code = {"f32": pa.PA_F32, "bf16": pa.PA_BF16, "e4m3": pa.PA_FP8_E4M3}[w.cache_dtype]
    if w.query_tile() and partition_size in (0, -1):
        # the query-tile kernel runs unsplit and uses no workspace
        return -1, 1, torch.zeros(16, dtype=torch.uint8, device=st.q.device)
    hq = w.Hq * w.nq   # varlen: query columns count as Hq * max_query_len heads
    P, nparts = pa.pa_decode_plan(w.S, hq, w.Hkv, w.D, w.max_blocks, code, 0, partition_size)
    nbytes = pa.pa_decode_workspace_size(w.S, hq, w.Hkv, w.D, w.max_blocks, P) \
        if (P > 0 or P == pa.PA_PARTITION_BALANCED) else 0
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=st.q.device)   # zero before first use
    return P, nparts, ws


def run_write(st: Staged) -> None:
    write_rows(st, st.k_step, st.v_step, st.slot_mapping)


def run_decode(st: Staged, partition_size: int = 0, ws=None, out=None) -> None:
    import paged_decode_attention_reshape_gb300 as pa
    w = st.w
    o = st.out if out is None else out
    ks, vs = (st.k_scale, st.v_scale) if st.fp8 else (None, None)
    if st.qsl is not None:
        pa.pa_attention_varlen(o, st.q, st.k_cache, st.v_cache, st.qsl, st.block_table, st.seq_lens, w.scale,
                               w.Hkv, w.nq, ks, vs, st.scale_stride, st.alibi, partition_size, ws, st.err)
    elif st.scale_stride or st.alibi is not None:
        pa.pa_decode_opt(o, st.q, st.k_cache, st.v_cache, st.block_table, st.seq_lens, w.scale, w.Hkv, ks, vs,
                         st.scale_stride, st.alibi, partition_size, ws, st.err)
    else:
        pa.pa_decode_ex(o, st.q, st.k_cache, st.v_cache, st.block_table, st.seq_lens, w.scale, w.Hkv, ks, vs,
                        partition_size, ws, st.err)


def run_step(st: Staged, partition_size: int = 0, ws=None) -> None:
    """One step of the hot path: the cache write of the step's rows, then attention.  A decode
    step whose rows are its sequences' newest tokens goes through pa_decode_step (one call; the
    decode reads the untouched pages while the write runs); otherwise two calls."""
    import paged_decode_attention_reshape_gb300 as pa
    nrs = getattr(st, "new_rows_start", False)
    if nrs is False:
        run_write(st)
        run_decode(st, partition_size, ws)
        return
    w = st.w
    ks, vs = (st.k_scale, st.v_scale) if st.fp8 else (None, None)
    pa.pa_decode_step(st.out, st.q, st.k_step, st.v_step, st.k_cache, st.v_cache, st.slot_mapping, st.block_table,
                      st.seq_lens, w.scale, w.Hkv, new_rows_start=nrs, k_scale=ks, v_scale=vs,
                      scale_stride=st.scale_stride, alibi_slopes=st.alibi, partition_size=partition_size,
                      workspace=ws, device_error=st.err)


# ------------------------------------------------------------ measurement

def _peaks(key="hbm_gbs"):
    """(peak, source): the measured HBM copy GB/s, or with key "bf16_tflops_sustained" the
    measured cuBLAS bf16 TFLOP/s of a seconds-long loop."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return (FALLBACK_HBM_GBS if key == "hbm_gbs" else FALLBACK_BF16_TFLOPS_SUSTAINED), "fallback"


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank space (string literals kept), so an edit to a
    comment does not count as a change of the kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':  # string literal, escapes included
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def decode_source_hash(sources=None) -> str:
    """Hash of the kernel sources' code (comments and spacing ignored): ncu traffic taken at
    another hash is reported as null."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_decode_attention_reshape_gb300", "csrc")
    for name in (sources or DECODE_SOURCES):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def _ncu_traffic(config: str, sources=None):
    """Per-launch DRAM bytes of the attention kernel from the committed ncu summary, if it was
    taken at the kernel's current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = decode_source_hash(sources)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == config and parts[1] == cur:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            self.uuid = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        def mine(r):
            return self.uuid is None or self.uuid in r[0] or r[0] in self.uuid
        rows = [r for (t, r) in self.rows if t0 <= t <= t1 and len(r) >= 9 and mine(r)]
        if len(rows) < 3:
            rows = [r for (t, r) in self.rows if len(r) >= 9 and mine(r)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.nanmedian(sm)), "sm_max_mhz": num(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": float(np.nanmax([num(r[3]) for r in rows]))}


def capture_step(st, partition_size, ws):
    """The step (write + attention) captured once in a CUDA graph: replaying it issues the
    same library launches, with their programmatic-launch edges, without per-launch host
    work -- the way a serving loop replays its decode step."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run_step(st, partition_size, ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def time_steps(st, K, flush, partition_size, ws, profile=False, graph=None):
    """Per-step device time (ms) of K steps, L2 flushed before each (outside the events);
    with `graph`, each step is a replay of the captured step."""
    import paged_decode_attention_reshape_gb300 as pa
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if profile:
        pa.pa_profile_read(pa.PA_KERNEL_WRITE)
        pa.pa_profile_read(pa.PA_KERNEL_DECODE)
        pa.pa_profile_enable(True)
    torch.cuda.synchronize()
    for i in range(K):
        flush()
        ev[i][0].record()
        torch.cuda.nvtx.range_push("step")
        if graph is not None:
            graph.replay()
        elif profile:
            # per-kernel times: the write and the attention as two calls, so the attention
            # kernel's time is its own (in pa_decode_step it starts early, while the write runs)
            run_write(st)
            run_decode(st, partition_size, ws)
        else:
            run_step(st, partition_size, ws)
        torch.cuda.nvtx.range_pop()
        ev[i][1].record()
    torch.cuda.synchronize()
    prof = None
    if profile:
        pa.pa_profile_enable(False)
        prof = {k: pa.pa_profile_read(k) for k in (pa.PA_KERNEL_WRITE, pa.PA_KERNEL_DECODE)}
    return [a.elapsed_time(b) for a, b in ev], prof


E2E_INPUTS = ("q", "k_step", "v_step", "slot_mapping", "block_table", "seq_lens")


def e2e_steps(st, K, flush, partition_size, ws):
    """Same step fed from host memory: the step's inputs (q, new K/V rows, slot_mapping,
    block_table, seq_lens) sit packed in one pinned host buffer, are copied to one device
    staging buffer (one H2D copy), the library runs on views of it, and the output comes
    back with one D2H copy, all inside the timed events."""
    import copy
    names = E2E_INPUTS + (("qsl",) if st.qsl is not None else ()) + \
        (("new_rows_start",) if isinstance(getattr(st, "new_rows_start", None), torch.Tensor) else ())
    offs, off = {}, 0
    for n in names:
        t = getattr(st, n)
        offs[n] = off
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev = torch.empty(off, dtype=torch.uint8, device=st.q.device)
    view = copy.copy(st)
    for n in names:
        t = getattr(st, n)
        nb = t.numel() * t.element_size()
        host[offs[n]:offs[n] + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        setattr(view, n, dev[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape))
    out_h = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    h2d = off
    d2h = out_h.numel() * out_h.element_size()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush()
        ev[i][0].record()
        dev.copy_(host, non_blocking=True)
        run_step(view, partition_size, ws)
        out_h.copy_(view.out, non_blocking=True)
        ev[i][1].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev], h2d, d2h


def cpu_baseline(w, target_s=12.0, max_seqs=None, threads=None):
    """Time the fp64 CPU oracle (as it stands) on a bounded sample of the workload: the cache
    write of the sampled sequences' step rows and the dense decode of all their query heads.
    Threads: one oracle call per (sequence) at a time on every host core (or `threads`)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    cores = threads or len(os.sched_getaffinity(0))
    rng = np.random.default_rng(7)
    order = rng.permutation(w.S)
    qs = data.q(w, "cpu").float().double().numpy().reshape(w.S, w.nq, w.Hq, w.D)

    def prep(s):
        K, V = data.logical_kv(w, int(s))
        if w.kv_dtype == "e4m3":   # bf16 bit patterns; the oracle quantises them itself
            return ("e4m3", K.view(torch.int16).numpy().view(np.uint16), V.view(torch.int16).numpy().view(np.uint16))
        return ("plain", K.float().numpy().astype(np.float64), V.float().numpy().astype(np.float64))

    def work(item):
        s, (kind, K, V) = item
        L = K.shape[0]
        if kind == "e4m3":
            ck = np.zeros((L, w.Hkv, w.D), dtype=np.uint8)
            cv = np.zeros((L, w.Hkv, w.D), dtype=np.uint8)
            oracle.write_flat(K, "bf16", np.arange(L), ck, "e4m3", w.k_scales())
            oracle.write_flat(V, "bf16", np.arange(L), cv, "e4m3", w.v_scales())
            K = oracle.cache_values(ck, "e4m3", w.k_scales())
            V = oracle.cache_values(cv, "e4m3", w.v_scales())
        if w.alibi is not None or w.nq > 1:
            oracle.attention_causal(qs[s], K, V, w.scale, w.alibi)
        else:
            oracle.dense_decode(qs[s][0], K, V, w.scale)
        return L

    # calibrate on one sequence, then size the sample to about target_s of wall time; a
    # workload the host finishes faster than that is run in repeated passes
    first = int(order[0])
    t = time.perf_counter()
    item0 = (first, prep(first))
    work(item0)
    one = time.perf_counter() - t
    n = int(max(1, min(w.S, (target_s * cores) / max(one, 1e-3))))
    if max_seqs:
        n = min(n, max_seqs)
    sample = [int(x) for x in order[:n]]
    items = [(s, prep(s)) for s in sample]
    passes = 0
    t = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while True:
            list(ex.map(work, items))
            passes += 1
            if time.perf_counter() - t >= target_s:
                break
    dt = time.perf_counter() - t
    nb = sum((int(w.seq_lens[s]) + 15) // 16 for s in sample)
    bytes_ = nb * 16 * w.Hkv * w.D * w.cache_elem_bytes() * 2 + 2 * n * w.nq * w.Hq * w.D * w.in_elem_bytes() + nb * 4 + n * 4
    return {"value": passes * bytes_ / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d pass(es) over %d of %d sequences (all %d query heads, fp64 dense decode%s), %.2f s"
                      % (passes, n, w.S, w.Hq, " + e4m3 quantisation" if w.kv_dtype == "e4m3" else "", dt),
            "tokens_per_s": passes * n * w.nq / dt}


# --------------------------------------------------------------------- main

def dist_setup(backend: str = "nccl"):
    """Rank layout from the torchrun environment.  Every rank works on its own GPU and its
    own batch (the path shards by sequence with no exchange), so the process group only
    carries the barrier and the max-over-ranks timing."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device="cuda"):
    if ws <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: int, ws: int, ms_max: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return ws * bytes_per_rank / (ms_max * 1e-3) / 1e9


def main_reference(args):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = configs.get(args.config)
    total_cpu_s = 150.0   # host seconds the whole reference run may take
    per_step = max(1.0, min(6.0, total_cpu_s / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(w, target_s=per_step / 3)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = cpu_baseline(w, target_s=per_step)
        vals.append(r)
    wall = time.perf_counter() - t0
    v = float(np.median([r["value"] for r in vals]))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": wall / max(1, args.steps) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name + " " + _workload_desc(w), "l2": "n/a (CPU)"},
            "cpu_baseline": {"kind": "oracle", "cores": vals[-1]["cores"], "sample": vals[-1]["sample"],
                             "value": v, "unit": "GB/s"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def _workload_desc(w):
    return ("S=%d Hq=%d Hkv=%d D=%d %s cache=%s L=[%d..%d] blocks=%d write_rows=%d"
            % (w.S, w.Hq, w.Hkv, w.D, w.dtype, w.cache_dtype, int(w.seq_lens.min()), int(w.seq_lens.max()),
               w.num_blocks, w.T))


# The workloads measured beside the headline one, each in the same JSON line: every decode
# workload of the configurations plus the chunked-prefill step on the query-tile kernel.
EXTRA_CONFIGS = ("c2", "c4", "c5", "c3-chunk128")


def measure(w, args, flush, sampler, ws=1, rank=0, cpu_target_s=12.0, partition_size=None, steps=None,
            e2e=True, soak_s=1.0):
    """Stage workload `w`, time K steps of the hot path on it and return its JSON fields.
    The step is captured in a CUDA graph and replayed K times (L2 flushed before each, outside
    the events); the same steps launched call by call, replayed warm (no flush), and a pass with
    the library's per-kernel profiling events give the other timings."""
    import paged_decode_attention_reshape_gb300 as pa
    dev = "cuda"
    K = args.steps if steps is None else steps
    part = args.partition_size if partition_size is None else partition_size
    st = stage(w, dev)
    P, nparts, wspace = workspace_for(st, part)
    for _ in range(args.warmup):
        flush()
        run_step(st, part, wspace)
    torch.cuda.synchronize()
    if sampler and soak_s > 0:
        # soak: keep the GPU busy so the sampled clocks are the loaded ones
        t_end = time.time() + soak_s
        while time.time() < t_end:
            for _ in range(20):
                flush()
                run_step(st, part, wspace)
            torch.cuda.synchronize()
    graph = capture_step(st, part, wspace)
    for _ in range(3):
        flush()
        graph.replay()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.time()
    step_ms, _ = time_steps(st, K, flush, part, wspace, profile=False, graph=graph)
    t1 = time.time()
    barrier(ws)
    # the same steps launched one call at a time from Python (reported beside the graph time)
    eager_ms, _ = time_steps(st, K, flush, part, wspace, profile=False)
    # and replayed back to back without the L2 flush (warm: what the previous step left in L2)
    warm_ms, _ = time_steps(st, K, lambda: None, part, wspace, profile=False, graph=graph)
    # per-kernel device times: the same steps again with the library's profiling events
    # around each launch (kept out of the step timing above: an event between the write and
    # the decode would hold back the decode's programmatic early launch)
    _, prof = time_steps(st, K, flush, part, wspace, profile=True)
    clocks = sampler.summary(t0 - 0.15, t1 + 0.15) if sampler else None
    rc, bits = pa.pa_check_device_error(st.err)
    if rc != 0:
        raise SystemExit("%s: device error word set: status %d bits %d" % (w.name, rc, bits))

    ms = max_over_ranks(float(np.mean(step_ms)), ws)
    eager = max_over_ranks(float(np.mean(eager_ms)), ws)
    warm = max_over_ranks(float(np.mean(warm_ms)), ws)
    pct = [float(x) for x in np.percentile(step_ms, [10, 50, 90])]
    dec_bytes = w.decode_bytes()
    value = job_throughput(dec_bytes, ws, ms)
    wr_ms, wr_n = prof[pa.PA_KERNEL_WRITE]
    dk_ms, dk_n = prof[pa.PA_KERNEL_DECODE]
    dk_avg = dk_ms / max(1, dk_n)
    peak, peak_src = _peaks()
    achieved = dec_bytes / (dk_avg * 1e-3) / 1e9
    if w.query_tile() and part in (0, -1):
        # tensor-bound: algorithmic FLOPs against the sustained bf16 peak (the kernel runs
        # inside a seconds-long loop of steps)
        flops = w.attention_flops()
        tpeak, tsrc = _peaks("bf16_tflops_sustained")
        tach = flops / (dk_avg * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": tach, "peak": tpeak, "unit": "TFLOP/s", "frac": tach / tpeak,
                    "traffic": _ncu_traffic(w.name, CHUNK_SOURCES), "peak_source": tsrc + " (sustained)",
                    "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": dec_bytes,
                    "hbm_GB/s": achieved, "kernel": "chunk_umma_kernel", "kernel_us": dk_avg * 1e3}
    else:
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "traffic": _ncu_traffic(w.name), "peak_source": peak_src,
                    "algorithmic_bytes_per_launch": dec_bytes, "kernel": "decode_mma_kernel",
                    "kernel_us": dk_avg * 1e3}

    e2e_d = None
    if e2e:
        e_ms, h2d, d2h = e2e_steps(st, max(10, min(K, 200)), flush, part, wspace)
        em = max_over_ranks(float(np.mean(e_ms)), ws)
        e2e_d = {"value": job_throughput(dec_bytes, ws, em), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h, "ms_per_step": em}
    del graph, st, wspace
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and cpu_target_s > 0:
        cpu = cpu_baseline(w, target_s=cpu_target_s)
        if w.S <= 64 and w.nq == 1:   # the small decode workloads: one host thread as well
            cpu["single_thread"] = cpu_baseline(w, target_s=min(4.0, cpu_target_s), threads=1)

    return {
        "value": value, "unit": "GB/s", "ms_per_step": ms, "steps": K,
        "config": {"workload": w.name + " " + _workload_desc(w),
                   "l2": "flushed before each step (512 MiB write + 512 MiB read)",
                   "partition_tokens": P, "partitions_max": nparts,
                   "parallelism": "replicas" if ws > 1 else "1 GPU"},
        "dtype": w.cache_dtype if w.cache_dtype != "auto" else w.dtype,
        "pct_of_hbm_peak": 100.0 * value / peak,
        "tokens_per_s": ws * w.S * w.nq / (ms * 1e-3),
        "step_ms_p10_p50_p90": pct,
        "eager_ms_per_step": eager, "eager_value": job_throughput(dec_bytes, ws, eager),
        "warm_ms_per_step": warm, "warm_value": job_throughput(dec_bytes, ws, warm),
        "decode_kernel_us": dk_avg * 1e3,
        "cache_write": {"GB/s": w.write_bytes() / ((wr_ms / max(1, wr_n)) * 1e-3) / 1e9,
                        "kernel_us": wr_ms / max(1, wr_n) * 1e3, "bytes": w.write_bytes()},
        "roofline": roofline,
        "gpu_launches": wr_n + dk_n,
        "clocks": clocks,
        "e2e": e2e_d,
        "cpu_baseline": cpu,
    }


# Partition sizes of the sweep (tokens; 0 = the library's plan, -1 = never split, -2 = the
# two-CTA cluster split, PA_PARTITION_BALANCED = the balanced split).
SWEEP = {"c4": [128, 256, 512, 1024, 2048, 4096, 8192, -2, -100, 0, -1],
         "c2": [256, 512, 1024, -2, -100, 0, -1],
         "c3": [512, 1024, 2048, -100, 0, -1],
         "c5": [512, 1024, 2048, -100, 0, -1]}


def sweep_partitions(args, flush):
    """Decode-kernel time of each workload at each partition size of SWEEP: the measurements
    the partition plan is fitted to.  Prints one JSON line per point and a Markdown table."""
    import paged_decode_attention_reshape_gb300 as pa
    names = args.sweep_configs.split(",") if args.sweep_configs else list(SWEEP)
    rows = []
    for name in names:
        w = configs.get(name)
        st = stage(w, "cuda")
        for part in SWEEP[name]:
            P, nparts, wspace = workspace_for(st, part)
            for _ in range(args.warmup):
                flush()
                run_step(st, part, wspace)
            _, prof = time_steps(st, args.steps, flush, part, wspace, profile=True)
            rc, bits = pa.pa_check_device_error(st.err)
            if rc != 0:
                raise SystemExit("%s P=%d: device error %d bits %d" % (name, part, rc, bits))
            dk_ms, dk_n = prof[pa.PA_KERNEL_DECODE]
            us = dk_ms / max(1, dk_n) * 1e3
            gbs = w.decode_bytes() / (us * 1e-6) / 1e9
            r = {"sweep": name, "request": part, "partition_tokens": P, "partitions_max": nparts,
                 "decode_kernel_us": us, "GB/s": gbs, "frac": gbs / _peaks()[0], "steps": dk_n}
            rows.append(r)
            print(json.dumps(r), flush=True)
            del wspace
        del st
        torch.cuda.empty_cache()
    label = {0: "plan", -1: "unsplit", -2: "cluster x2", -100: "balanced"}
    print("| workload | request | partition (tokens) | partitions | decode kernel (us) | GB/s | frac of measured peak |")
    print("|---|---|---|---|---|---|---|")
    for r in rows:
        req = label.get(r["request"], str(r["request"]))
        pt = {0: "unsplit", -100: "balanced"}.get(r["partition_tokens"], str(r["partition_tokens"]))
        print("| %s | %s | %s | %d | %.1f | %.0f | %.3f |" % (r["sweep"], req, pt, r["partitions_max"],
                                                            r["decode_kernel_us"], r["GB/s"], r["frac"]))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="c3", choices=sorted(configs.BUILDERS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--extra-configs", default=",".join(EXTRA_CONFIGS),
                    help="workloads measured beside the headline one, in the same line ('' for none)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="setup + warm-up steps only (profiling runs)")
    ap.add_argument("--no-soak", action="store_true", help="skip the 1 s clock soak before the timed steps")
    ap.add_argument("--sweep-partitions", action="store_true",
                    help="time the decode kernel over the partition sizes the plan is fitted to")
    ap.add_argument("--sweep-configs", default="", help="workloads of the sweep (default: all)")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return main_reference(args)
    if args.warmup < 3:
        args.warmup = 3

    import paged_decode_attention_reshape_gb300 as pa
    pa.lib()
    ws, rank, local = dist_setup()
    flush = L2Flush("cuda")
    if args.sweep_partitions:
        return sweep_partitions(args, flush)
    w = configs.get(args.config)
    if args.quick:
        st = stage(w, "cuda")
        P, nparts, wspace = workspace_for(st, args.partition_size)
        for _ in range(args.warmup):
            flush()
            run_step(st, args.partition_size, wspace)
        torch.cuda.synchronize()
        rc, bits = pa.pa_check_device_error(st.err)
        if rc != 0:
            raise SystemExit("device error %d bits %d" % (rc, bits))
        print(json.dumps({"quick": True, "config": w.name, "partition": P}), flush=True)
        return 0

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    soak = 0.0 if args.no_soak else 1.0
    main_m = measure(w, args, flush, sampler, ws, rank, cpu_target_s=0 if args.no_cpu_baseline else 12.0,
                     e2e=not args.no_e2e, soak_s=soak)
    extras = {}
    for name in [n for n in args.extra_configs.split(",") if n and n != args.config]:
        # the other workloads: the same measurement, the default partition plan, a shorter
        # CPU-oracle sample
        extras[name] = measure(configs.get(name), args, flush, sampler, ws, rank,
                               cpu_target_s=0 if args.no_cpu_baseline else 4.0, partition_size=0,
                               e2e=not args.no_e2e, soak_s=min(soak, 0.3))
    if sampler:
        sampler.stop()

    line = {
        "metric": METRIC, "value": main_m["value"], "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main_m["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": main_m["dtype"], "data": "synthetic",
        "config": main_m["config"],
        "launch": "step replayed from a CUDA graph (write + attention, programmatic-launch edge kept)",
    }
    for k in ("pct_of_hbm_peak", "tokens_per_s", "step_ms_p10_p50_p90", "eager_ms_per_step", "eager_value",
              "warm_ms_per_step", "warm_value", "decode_kernel_us", "cache_write", "roofline", "gpu_launches",
              "clocks", "e2e", "cpu_baseline"):
        line[k] = main_m[k]
    if extras:
        line["configs"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
