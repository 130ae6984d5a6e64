"""Host logic of bench.py that needs no GPU: how a workload's step rows map to sequences for
pa_decode_step, and the workloads' algorithmic FLOP counts and kernel choice."""
import numpy as np
import torch

import bench
from workloads import configs


def test_one_new_token_per_sequence_needs_no_row_starts():
    for name in ("c1", "c2", "c3", "c4", "c2-nhd", "c3-alibi"):
        w = configs.get(name)
        if name == "c1":   # c1's step writes six rows (one padding) for two sequences
            assert bench.new_rows_start(w, "cpu") is False
            continue
        assert bench.new_rows_start(w, "cpu") is None, name


def test_chunk_rows_give_row_starts():
    """c5 writes the last 64 positions of each sequence, sequence after sequence."""
    for name in ("c5", "c5-heads"):
        w = configs.get(name)
        nrs = bench.new_rows_start(w, "cpu")
        assert isinstance(nrs, torch.Tensor) and nrs.dtype == torch.int32
        assert nrs.tolist() == list(range(0, 64 * w.S + 1, 64))


def test_multi_query_steps_keep_two_calls():
    for name in ("c3-spec4", "c3-chunk128"):
        assert bench.new_rows_start(configs.get(name), "cpu") is False


def test_rows_out_of_order_keep_two_calls():
    w = configs.get("c5")
    w.step_seq = w.step_seq[::-1].copy()
    w.step_pos = w.step_pos[::-1].copy()
    assert bench.new_rows_start(w, "cpu") is False


def test_attention_flops_brute_force():
    """4 D Hq per visible (query, key) pair, counted by brute force on a small case."""
    w = configs.get("c3-spec4")
    w.seq_lens = np.array([5, 9, 4], dtype=np.int32)
    w.S = 3
    pairs = 0
    for L in w.seq_lens:
        for i in range(w.nq):
            pos = int(L) - w.nq + i
            pairs += pos + 1
    assert w.attention_flops() == 4.0 * w.D * w.Hq * pairs


def test_query_tile_choice():
    assert configs.get("c3-chunk128").query_tile()
    assert not configs.get("c3-spec4").query_tile()   # 16 query columns per KV head
    assert not configs.get("c3").query_tile()
    assert not configs.get("c5").query_tile()         # one query token per sequence


def test_source_hash_ignores_comments_and_spacing_only():
    code = 'int a = 1;  // note\n/* block\n comment */ asm("mov.u32 %0, %1; // not a comment");\nint b;'
    same = 'int a = 1;\n\n   asm("mov.u32 %0, %1; // not a comment"); int b;'
    other = 'int a = 2; asm("mov.u32 %0, %1; // not a comment"); int b;'
    lit = 'int a = 1; asm("mov.u32 %0, %1; // another literal"); int b;'
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)
    assert bench._code_only(code) != bench._code_only(lit)     # text inside a string literal counts
    assert bench._code_only('s = "a \\" // b"; x;') == 's = "a \\" // b"; x;'
