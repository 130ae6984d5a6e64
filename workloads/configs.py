"""The five synthetic workloads, as metadata plus seeded value streams.

Each builder returns a ``Workload``: shapes, dtypes, sequence lengths, block
tables and the rows written in the measured step.  Values are not stored: both
sides regenerate them from ``workloads.gen`` with the workload's seed.

This module stands in for the serving engine upstream of the hot path: it
allocates physical blocks (a seeded permutation of the pool, as a block
manager would hand them out) and produces the metadata the kernels consume --
``block_table``, ``seq_lens`` and ``slot_mapping``.  A position's slot is the
flat index its allocator-assigned block gives it,
``block_table[s][pos // block_size] * block_size + pos % block_size``; that is
how the slot-mapping metadata is defined upstream of the write ("How vLLM CUDA
Kernels Write and Read the Paged KV Cache", "Mapping one token to a physical
slot").  Nothing here touches K/V values or attention.

Recipes (seed = 0x5EED0000 + config index):

c1  tiny MHA fp32: S=2, Hq=Hkv=4, D=64, 16-block pool, L={5,37}; sequence 1
    owns blocks [7,2,9] (position 20 -> slot 36), sequence 0 one block from a
    seeded shuffle of the other 13; step rows (s0,4) (s1,20) (s1,33) (s1,34)
    (s1,36) and one padding row (slot -1, NaN data); scale 1/8.
c2  S=64, 32/8 heads, D=64, bf16, pool 65536 blocks, L ~ U{1..2048}; one new
    token per sequence (position L-1).
c3  S=256, 32/8, D=128, bf16, L ~ U{512..4096}, pool ceil(1.25 x needed).
c4  S=4, 32/8, D=128, bf16, L = {32768, 65536, 98304, 131072}, pool 1.25x;
    one outlier key per sequence whose logit for the first query head of each
    KV group is about +20; one new token per sequence.
c5  write: 8192 rows = the last 64 positions of 128 sequences, 5% of them
    padding (slot -1; those positions keep their earlier values), bf16 ->
    fp8 e4m3 with k_scale = v_scale = 0.05; decode S=128, 64/8 heads, D=128,
    L ~ U{1024..8192}, pool 1.25x.

Variants with the same values: c2-nhd (NHD cache layout), c3-alibi (ALiBi
slopes), c5-heads (one FP8 scale per KV head), c3-spec4 (4 query tokens per
sequence, varlen attention; the first token's q is c3's), c3-chunk128 (128 new tokens
per sequence: a chunked-prefill step).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 16


@dataclass
class Workload:
    name: str
    seed: int
    S: int
    Hq: int
    Hkv: int
    D: int
    dtype: str             # q / new-row / output dtype: "f32" or "bf16"
    kv_dtype: str          # cache element: "auto" (same as dtype) or "e4m3"
    scale: float
    k_scale: float
    v_scale: float
    num_blocks: int
    seq_lens: np.ndarray   # int32 [S]
    block_table: np.ndarray  # int32 [S, max_blocks]; entries past ceil(L/16) are padding
    step_seq: np.ndarray   # int64 [T]: sequence of each step row (-1 for padding rows)
    step_pos: np.ndarray   # int64 [T]: position of each step row
    step_slot: np.ndarray  # int64 [T]: slot_mapping of the step (-1 = padding)
    outlier_pos: np.ndarray | None = None  # int64 [S] (c4) or None
    notes: dict = field(default_factory=dict)
    layout: str = "hnd"                    # cache layout: "hnd" [NB, Hkv, 16, D] or "nhd" [NB, 16, Hkv, D]
    k_head_scales: np.ndarray | None = None  # fp32 [Hkv]: per-head FP8 scales (replace k_scale / v_scale)
    v_head_scales: np.ndarray | None = None
    alibi: np.ndarray | None = None        # fp32 [Hq]: ALiBi slopes, or None
    nq: int = 1                            # new query tokens per sequence (> 1: varlen attention)

    def k_scales(self):
        """The K quantisation scale(s) the write uses: one float, or [Hkv] per-head scales."""
        return self.k_scale if self.k_head_scales is None else self.k_head_scales

    def v_scales(self):
        return self.v_scale if self.v_head_scales is None else self.v_head_scales

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def cache_dtype(self) -> str:
        return self.dtype if self.kv_dtype == "auto" else self.kv_dtype

    @property
    def T(self) -> int:
        return int(self.step_slot.shape[0])

    def n_blocks_of(self, s: int) -> int:
        return (int(self.seq_lens[s]) + BLOCK - 1) // BLOCK

    def slot_of(self, s: int, pos) -> np.ndarray:
        pos = np.asarray(pos, dtype=np.int64)
        return self.block_table[s][pos // BLOCK].astype(np.int64) * BLOCK + pos % BLOCK

    def step_written(self) -> set:
        """(seq, pos) pairs overwritten by the step (padding rows excluded)."""
        return {(int(s), int(p)) for s, p, sl in zip(self.step_seq, self.step_pos, self.step_slot) if sl >= 0}

    def cache_elem_bytes(self) -> int:
        return {"f32": 4, "bf16": 2, "e4m3": 1}[self.cache_dtype]

    def in_elem_bytes(self) -> int:
        return {"f32": 4, "bf16": 2}[self.dtype]

    def decode_bytes(self) -> int:
        """Algorithmic bytes of one decode call: K+V pages touched once per KV head,
        plus q, out, the block-table entries read, seq_lens (and query_start_loc)."""
        nb = sum(self.n_blocks_of(s) for s in range(self.S))
        kv = nb * BLOCK * self.Hkv * self.D * self.cache_elem_bytes() * 2
        qo = 2 * self.S * self.nq * self.Hq * self.D * self.in_elem_bytes()
        qsl = (self.S + 1) * 4 if self.nq > 1 else 0
        return kv + qo + nb * 4 + self.S * 4 + qsl

    def attention_flops(self) -> float:
        """Algorithmic FLOPs of one attention call: q.k and p.v, 2 D each, for every (query
        head, visible key) pair; new token i of n sits at position L - n + i and sees i + 1
        + (L - n) keys."""
        n = self.nq
        pairs = sum(n * int(L) - n * (n - 1) // 2 for L in self.seq_lens)
        return 4.0 * self.D * self.Hq * pairs

    def query_tile(self) -> bool:
        """True when attention runs on the query-tile tensor-core kernel: 64 or more query
        columns (new tokens x G) per KV head (32 at head size 64), a 16-bit cache, head size
        64 or 128."""
        return (self.nq > 1 and self.nq * self.G >= (32 if self.D == 64 else 64)
                and self.cache_dtype in ("bf16", "f16") and self.D in (64, 128))

    def write_bytes(self) -> int:
        """Algorithmic bytes of one cache write: valid rows read and written, plus slot_mapping."""
        valid = int((self.step_slot >= 0).sum())
        return valid * self.Hkv * self.D * (self.in_elem_bytes() + self.cache_elem_bytes()) * 2 + self.T * 8


def _tables(rng, lens, num_blocks, max_blocks):
    """Assign each sequence's blocks from a seeded permutation of the pool."""
    need = [(int(L) + BLOCK - 1) // BLOCK for L in lens]
    assert sum(need) <= num_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    o = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[o:o + n]
        o += n
    return bt


def _decode_step(w_seq_lens):
    S = len(w_seq_lens)
    seqs = np.arange(S, dtype=np.int64)
    pos = np.asarray(w_seq_lens, dtype=np.int64) - 1
    return seqs, pos


def c1() -> Workload:
    seed = 0x5EED0000
    rng = np.random.default_rng(seed)
    lens = np.array([5, 37], dtype=np.int32)
    bt = np.full((2, 3), -1, dtype=np.int32)
    bt[1] = [7, 2, 9]
    others = np.array([b for b in range(16) if b not in (7, 2, 9)], dtype=np.int32)
    bt[0, 0] = rng.permutation(others)[0]
    w = Workload("c1", seed, 2, 4, 4, 64, "f32", "auto", 1.0 / 8.0, 1.0, 1.0, 16, lens, bt,
                 np.array([0, 1, 1, 1, 1, -1], dtype=np.int64),
                 np.array([4, 20, 33, 34, 36, 0], dtype=np.int64),
                 np.zeros(6, dtype=np.int64))
    w.step_slot = np.array([int(w.slot_of(int(s), int(p))) if s >= 0 else -1
                            for s, p in zip(w.step_seq, w.step_pos)], dtype=np.int64)
    return w


def c2() -> Workload:
    seed = 0x5EED0001
    rng = np.random.default_rng(seed)
    S, NB = 64, 65536
    lens = rng.integers(1, 2048, size=S, endpoint=True).astype(np.int32)
    bt = _tables(rng, lens, NB, 2048 // BLOCK)
    seqs, pos = _decode_step(lens)
    w = Workload("c2", seed, S, 32, 8, 64, "bf16", "auto", 1.0 / math.sqrt(64), 1.0, 1.0, NB, lens, bt,
                 seqs, pos, np.zeros(S, dtype=np.int64))
    w.step_slot = np.array([int(w.slot_of(int(s), int(p))) for s, p in zip(seqs, pos)], dtype=np.int64)
    return w


def _pool(lens):
    need = sum((int(L) + BLOCK - 1) // BLOCK for L in lens)
    return int(math.ceil(1.25 * need))


def c3() -> Workload:
    seed = 0x5EED0002
    rng = np.random.default_rng(seed)
    S = 256
    lens = rng.integers(512, 4096, size=S, endpoint=True).astype(np.int32)
    NB = _pool(lens)
    bt = _tables(rng, lens, NB, 4096 // BLOCK)
    seqs, pos = _decode_step(lens)
    w = Workload("c3", seed, S, 32, 8, 128, "bf16", "auto", 1.0 / math.sqrt(128), 1.0, 1.0, NB, lens, bt,
                 seqs, pos, np.zeros(S, dtype=np.int64))
    w.step_slot = np.array([int(w.slot_of(int(s), int(p))) for s, p in zip(seqs, pos)], dtype=np.int64)
    return w


def c4() -> Workload:
    seed = 0x5EED0003
    rng = np.random.default_rng(seed)
    lens = np.array([32768, 65536, 98304, 131072], dtype=np.int32)
    NB = _pool(lens)
    bt = _tables(rng, lens, NB, 131072 // BLOCK)
    seqs, pos = _decode_step(lens)
    # one outlier position per sequence, away from the step row
    outl = np.array([int(rng.integers(0, int(L) - 1)) for L in lens], dtype=np.int64)
    w = Workload("c4", seed, 4, 32, 8, 128, "bf16", "auto", 1.0 / math.sqrt(128), 1.0, 1.0, NB, lens, bt,
                 seqs, pos, np.zeros(4, dtype=np.int64), outlier_pos=outl)
    w.step_slot = np.array([int(w.slot_of(int(s), int(p))) for s, p in zip(seqs, pos)], dtype=np.int64)
    w.notes["outlier_logit"] = 20.0
    return w


def c5() -> Workload:
    seed = 0x5EED0004
    rng = np.random.default_rng(seed)
    S = 128
    lens = rng.integers(1024, 8192, size=S, endpoint=True).astype(np.int32)
    NB = _pool(lens)
    bt = _tables(rng, lens, NB, 8192 // BLOCK)
    per = 64
    seqs = np.repeat(np.arange(S, dtype=np.int64), per)
    pos = np.concatenate([np.arange(int(L) - per, int(L), dtype=np.int64) for L in lens])
    T = S * per
    pad = np.zeros(T, dtype=bool)
    pad[rng.choice(T, size=int(round(0.05 * T)), replace=False)] = True
    w = Workload("c5", seed, S, 64, 8, 128, "bf16", "e4m3", 1.0 / math.sqrt(128), 0.05, 0.05, NB, lens, bt,
                 seqs, pos, np.zeros(T, dtype=np.int64))
    slots = np.concatenate([w.slot_of(s, pos[s * per:(s + 1) * per]) for s in range(S)])
    slots[pad] = -1
    w.step_slot = slots.astype(np.int64)
    w.notes["padding_rows"] = int(pad.sum())
    return w


def c2_nhd() -> Workload:
    """c2 with the caches token-major within a block ([NB, 16, Hkv, D], the NHD layout of
    "Inside vLLM CUDA Kernels", Part 2); same values."""
    w = c2()
    w.name, w.layout = "c2-nhd", "nhd"
    return w


def c3_alibi() -> Workload:
    """c3 with ALiBi: head h of 32 gets slope 2^(-8 (h + 1) / 32), the usual geometric slopes."""
    w = c3()
    w.name = "c3-alibi"
    w.alibi = (2.0 ** (-8.0 * np.arange(1, w.Hq + 1) / w.Hq)).astype(np.float32)
    return w


def c5_heads() -> Workload:
    """c5 with one FP8 scale per KV head: K heads 0.04, 0.045, ..., 0.075; V heads the reverse
    order (|x| / scale stays below 4.5 / 0.04 < 448: no saturation)."""
    w = c5()
    w.name = "c5-heads"
    w.k_head_scales = (0.04 + 0.005 * np.arange(w.Hkv)).astype(np.float32)
    w.v_head_scales = w.k_head_scales[::-1].copy()
    return w


def c3_spec4() -> Workload:
    """c3 with 4 new query tokens per sequence (speculative decoding: one token plus three
    draft tokens): the step writes each sequence's last 4 positions and attends causally."""
    return _c3_new_tokens("c3-spec4", 4)


def c3_chunk128() -> Workload:
    """c3 as one chunked-prefill step: the last 128 positions of each of the 256 sequences are
    new (32768 rows written), every new token attends causally to its history and the chunk
    -- 512 query rows per KV head, the query-tile tensor-core kernel's case."""
    return _c3_new_tokens("c3-chunk128", 128)


def _c3_new_tokens(name: str, nq: int) -> Workload:
    w = c3()
    w.name, w.nq = name, nq
    seqs = np.repeat(np.arange(w.S, dtype=np.int64), w.nq)
    pos = np.concatenate([np.arange(int(L) - w.nq, int(L), dtype=np.int64) for L in w.seq_lens])
    w.step_seq, w.step_pos = seqs, pos
    w.step_slot = np.concatenate([w.slot_of(s, pos[s * w.nq:(s + 1) * w.nq]) for s in range(w.S)]).astype(np.int64)
    return w


BUILDERS = {"c1": c1, "c2": c2, "c3": c3, "c4": c4, "c5": c5, "c2-nhd": c2_nhd, "c3-alibi": c3_alibi,
            "c5-heads": c5_heads, "c3-spec4": c3_spec4, "c3-chunk128": c3_chunk128}


def get(name: str) -> Workload:
    return BUILDERS[name]()
