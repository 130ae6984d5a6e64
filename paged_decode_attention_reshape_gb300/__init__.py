"""Python binding of libpa_gb300.so (include/pa.h): argument marshalling only.

Every function here turns torch tensors into ``pa_tensor`` descriptors (data
pointer, element type, extents, strides) and calls the C ABI function of the
same name on the current CUDA stream.  No computation happens in Python, and
there is no fallback: if the library is not built, importing works but the
first call raises ``RuntimeError``.

Element types: float32, bfloat16, float16; E4M3 caches as torch.uint8 (raw
codes) or torch.float8_e4m3fn; block tables and sequence lengths int32;
slot_mapping int64.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa_gb300.so")

PA_F32, PA_BF16, PA_F16, PA_FP8_E4M3, PA_I32, PA_I64 = range(6)
PA_KV_AUTO, PA_KV_FP8_E4M3 = 0, 1
PA_KERNEL_WRITE, PA_KERNEL_DECODE = 0, 1
PA_DEVERR_SLOT_RANGE, PA_DEVERR_BLOCK_RANGE, PA_DEVERR_SEQLEN_RANGE, PA_DEVERR_WAIT_TIMEOUT = 1, 2, 4, 8
STATUS = {0: "PA_OK", -1: "PA_ERR_INVALID_ARG", -2: "PA_ERR_UNSUPPORTED_DTYPE", -3: "PA_ERR_ALIGNMENT",
          -4: "PA_ERR_WORKSPACE", -5: "PA_ERR_CUDA", -6: "PA_ERR_DEVICE_BOUNDS", -7: "PA_ERR_UNSUPPORTED_SHAPE",
          -8: "PA_ERR_DEVICE_TIMEOUT", -9: "PA_ERR_NO_BLOCKS"}

EXPORTS = ("pa_reshape_and_cache", "pa_reshape_and_cache_opt", "pa_decode", "pa_decode_ex", "pa_decode_opt",
           "pa_attention_varlen", "pa_decode_step", "pa_decode_noalloc", "pa_decode_plan", "pa_decode_workspace_size", "pa_check_device_error",
           "pa_status_string", "pa_profile_enable", "pa_profile_read", "pa_bm_create", "pa_bm_destroy",
           "pa_bm_num_free", "pa_bm_block_refs", "pa_bm_seq_len", "pa_bm_append", "pa_bm_fork", "pa_bm_free",
           "pa_bm_export", "pa_copy_blocks")
PA_NOALLOC_SCRATCH_BYTES = 32 << 20
PA_PARTITION_BALANCED = -100  # partition_size: balanced split over one resident wave

_DT = {torch.float32: PA_F32, torch.bfloat16: PA_BF16, torch.float16: PA_F16, torch.uint8: PA_FP8_E4M3,
       torch.int32: PA_I32, torch.int64: PA_I64}
if hasattr(torch, "float8_e4m3fn"):
    _DT[torch.float8_e4m3fn] = PA_FP8_E4M3


class PaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5), ("stride", ctypes.c_int64 * 5)]


class PaWriteOptions(ctypes.Structure):
    _fields_ = [("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("scale_stride", ctypes.c_int64),
                ("device_error", ctypes.c_void_p)]


class PaDecodeOptions(ctypes.Structure):
    _fields_ = [("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("scale_stride", ctypes.c_int64),
                ("alibi_slopes", ctypes.c_void_p), ("partition_size", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("device_error", ctypes.c_void_p), ("first_wait_limit", ctypes.c_int)]


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (where, STATUS.get(status, status), status_string(status)))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libpa_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libpa_gb300.so is not built (expected at %s); run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            P, T = ctypes.c_void_p, ctypes.POINTER(PaTensor)
            i32, f32 = ctypes.c_int, ctypes.c_float
            L.pa_reshape_and_cache.restype = i32
            L.pa_reshape_and_cache.argtypes = [T, T, T, T, T, i32, P, P, P, P]
            L.pa_reshape_and_cache_opt.restype = i32
            L.pa_reshape_and_cache_opt.argtypes = [T, T, T, T, T, i32, ctypes.POINTER(PaWriteOptions), P]
            L.pa_decode_opt.restype = i32
            L.pa_decode_opt.argtypes = [T, T, T, T, T, T, f32, i32, ctypes.POINTER(PaDecodeOptions), P]
            L.pa_decode_step.restype = i32
            L.pa_decode_step.argtypes = [T, T, T, T, T, T, T, T, T, T, f32, i32, ctypes.POINTER(PaDecodeOptions), P]
            L.pa_attention_varlen.restype = i32
            L.pa_attention_varlen.argtypes = [T, T, T, T, T, T, T, f32, i32, i32, ctypes.POINTER(PaDecodeOptions), P]
            i64p = ctypes.POINTER(ctypes.c_int64)
            L.pa_bm_create.restype = P
            L.pa_bm_create.argtypes = [i32, i32, i32]
            L.pa_bm_destroy.restype = None
            L.pa_bm_destroy.argtypes = [P]
            L.pa_bm_num_free.restype = i32
            L.pa_bm_num_free.argtypes = [P]
            L.pa_bm_block_refs.restype = i32
            L.pa_bm_block_refs.argtypes = [P, i32]
            L.pa_bm_seq_len.restype = ctypes.c_int64
            L.pa_bm_seq_len.argtypes = [P, i32]
            L.pa_bm_append.restype = i32
            L.pa_bm_append.argtypes = [P, i32, i32, i64p, i64p, ctypes.POINTER(i32)]
            L.pa_bm_fork.restype = i32
            L.pa_bm_fork.argtypes = [P, i32, i32]
            L.pa_bm_free.restype = i32
            L.pa_bm_free.argtypes = [P, i32]
            L.pa_bm_export.restype = i32
            L.pa_bm_export.argtypes = [P, ctypes.POINTER(i32), i32, i32, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int32)]
            L.pa_copy_blocks.restype = i32
            L.pa_copy_blocks.argtypes = [T, T, T, P, P]
            L.pa_decode.restype = i32
            L.pa_decode.argtypes = [T, T, T, T, T, T, f32, i32, P]
            L.pa_decode_ex.restype = i32
            L.pa_decode_ex.argtypes = [T, T, T, T, T, T, f32, i32, P, P, i32, P, ctypes.c_size_t, P, P]
            L.pa_decode_noalloc.restype = i32
            L.pa_decode_noalloc.argtypes = [T, T, T, T, T, T, f32, i32, P, P, i32, P, P]
            L.pa_decode_plan.restype = i32
            L.pa_decode_plan.argtypes = [i32] * 8 + [ctypes.POINTER(i32), ctypes.POINTER(i32)]
            L.pa_decode_workspace_size.restype = ctypes.c_size_t
            L.pa_decode_workspace_size.argtypes = [i32] * 6
            L.pa_check_device_error.restype = i32
            L.pa_check_device_error.argtypes = [P, ctypes.POINTER(i32), P]
            L.pa_status_string.restype = ctypes.c_char_p
            L.pa_status_string.argtypes = [i32]
            L.pa_profile_enable.restype = i32
            L.pa_profile_enable.argtypes = [i32]
            L.pa_profile_read.restype = i32
            L.pa_profile_read.argtypes = [i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong)]
            _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().pa_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS.get(status, "unknown")


def desc(t: torch.Tensor, dtype_code: int | None = None) -> PaTensor:
    """pa_tensor for a torch tensor (no copy)."""
    if t.dim() > 5:
        raise ValueError("rank > 5")
    d = PaTensor()
    d.data = t.data_ptr() if t.numel() else 0
    d.dtype = _DT[t.dtype] if dtype_code is None else dtype_code
    d.ndim = t.dim()
    for i, (n, s) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = n
        d.stride[i] = s
    return d


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(rc: int, where: str):
    if rc != 0:
        raise PAError(rc, where)


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, kv_dtype: int = PA_KV_AUTO,
                         k_scale=None, v_scale=None, device_error=None, stream=None) -> None:
    """Scatter key/value [T, Hkv, D] rows into k_cache/v_cache [NB, Hkv, 16, D] at slot_mapping [T] (int64).
    kv_dtype PA_KV_FP8_E4M3 quantises with the device fp32 scales k_scale/v_scale (1-element tensors)."""
    args = (desc(key), desc(value), desc(k_cache), desc(v_cache), desc(slot_mapping))
    rc = lib().pa_reshape_and_cache(*[ctypes.byref(a) for a in args], int(kv_dtype), _ptr(k_scale), _ptr(v_scale),
                                    _ptr(device_error), _stream(stream))
    _check(rc, "pa_reshape_and_cache")


def pa_reshape_and_cache_opt(key, value, k_cache, v_cache, slot_mapping, kv_dtype: int = PA_KV_AUTO,
                             k_scale=None, v_scale=None, scale_stride: int = 0, device_error=None,
                             stream=None) -> None:
    """pa_reshape_and_cache with per-head FP8 scales: KV head h uses k_scale[h * scale_stride]
    (scale_stride 0: one scale for every head).  The cache may be a strided view (an NHD cache
    [NB, 16, Hkv, D] passed as .permute(0, 2, 1, 3))."""
    o = PaWriteOptions(_ptr(k_scale), _ptr(v_scale), int(scale_stride), _ptr(device_error))
    args = (desc(key), desc(value), desc(k_cache), desc(v_cache), desc(slot_mapping))
    rc = lib().pa_reshape_and_cache_opt(*[ctypes.byref(a) for a in args], int(kv_dtype), ctypes.byref(o),
                                        _stream(stream))
    _check(rc, "pa_reshape_and_cache_opt")


def pa_decode_opt(out, q, k_cache, v_cache, block_table, seq_lens, scale: float, num_kv_heads: int,
                  k_scale=None, v_scale=None, scale_stride: int = 0, alibi_slopes=None, partition_size: int = 0,
                  workspace=None, device_error=None, stream=None, first_wait_limit: int = 0) -> None:
    """pa_decode with every option: per-head FP8 scales (KV head h uses k_scale[h * scale_stride]),
    ALiBi slopes (fp32 [Hq]: logit += slope_h * (t - (seq_len - 1))), partition size, caller
    workspace (None: the library's internal one) and device error word.  first_wait_limit: poll
    limit of the first pipeline wait (0 normal, < 0 give up at once), for testing the timeout path."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    o = PaDecodeOptions(_ptr(k_scale), _ptr(v_scale), int(scale_stride), _ptr(alibi_slopes), int(partition_size),
                        _ptr(workspace), ws_bytes, _ptr(device_error), int(first_wait_limit))
    args = (desc(out), desc(q), desc(k_cache), desc(v_cache), desc(block_table), desc(seq_lens))
    rc = lib().pa_decode_opt(*[ctypes.byref(a) for a in args], float(scale), int(num_kv_heads), ctypes.byref(o),
                             _stream(stream))
    _check(rc, "pa_decode_opt")


def pa_decode_step(out, q, key, value, k_cache, v_cache, slot_mapping, block_table, seq_lens, scale: float,
                   num_kv_heads: int, new_rows_start=None, k_scale=None, v_scale=None, scale_stride: int = 0,
                   alibi_slopes=None, partition_size: int = 0, workspace=None, device_error=None,
                   stream=None, first_wait_limit: int = 0) -> None:
    """The cache write of the step's new rows (key / value [T, Hkv, D] to slot_mapping) and the
    decode over the updated cache in one call; the decode reads everything but the new
    positions while the write runs.  new_rows_start: None (row s = sequence s's newest token)
    or int32 [S+1] (rows of sequence s, its newest tokens in order).  Options as pa_decode_opt;
    the scales also quantise the rows written to an FP8 cache."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    o = PaDecodeOptions(_ptr(k_scale), _ptr(v_scale), int(scale_stride), _ptr(alibi_slopes), int(partition_size),
                        _ptr(workspace), ws_bytes, _ptr(device_error), int(first_wait_limit))
    nrs = None if new_rows_start is None else ctypes.byref(desc(new_rows_start))
    args = (desc(out), desc(q), desc(key), desc(value), desc(k_cache), desc(v_cache), desc(slot_mapping))
    rc = lib().pa_decode_step(*[ctypes.byref(a) for a in args], nrs, ctypes.byref(desc(block_table)),
                              ctypes.byref(desc(seq_lens)), float(scale), int(num_kv_heads), ctypes.byref(o),
                              _stream(stream))
    _check(rc, "pa_decode_step")


def pa_attention_varlen(out, q, k_cache, v_cache, query_start_loc, block_table, seq_lens, scale: float,
                        num_kv_heads: int, max_query_len: int, k_scale=None, v_scale=None, scale_stride: int = 0,
                        alibi_slopes=None, partition_size: int = 0, workspace=None, device_error=None,
                        stream=None, first_wait_limit: int = 0) -> None:
    """Several new query tokens per sequence: q/out [Tq, Hq, D] packed, sequence s owning rows
    query_start_loc[s] .. query_start_loc[s+1]-1 (int32 [S+1]); query i of s sits at position
    seq_lens[s] - n_s + i and sees the tokens up to it.  Options as pa_decode_opt; the workspace
    size is pa_decode_workspace_size with num_heads = Hq * max_query_len."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    o = PaDecodeOptions(_ptr(k_scale), _ptr(v_scale), int(scale_stride), _ptr(alibi_slopes), int(partition_size),
                        _ptr(workspace), ws_bytes, _ptr(device_error), int(first_wait_limit))
    args = (desc(out), desc(q), desc(k_cache), desc(v_cache), desc(query_start_loc), desc(block_table),
            desc(seq_lens))
    rc = lib().pa_attention_varlen(*[ctypes.byref(a) for a in args], float(scale), int(num_kv_heads),
                                   int(max_query_len), ctypes.byref(o), _stream(stream))
    _check(rc, "pa_attention_varlen")


def pa_decode(out, q, k_cache, v_cache, block_table, seq_lens, scale: float, num_kv_heads: int,
              stream=None) -> None:
    """Paged decode attention: out/q [S, Hq, D], caches [NB, Hkv, 16, D], block_table [S, maxNB] int32,
    seq_lens [S] int32."""
    args = (desc(out), desc(q), desc(k_cache), desc(v_cache), desc(block_table), desc(seq_lens))
    rc = lib().pa_decode(*[ctypes.byref(a) for a in args], float(scale), int(num_kv_heads), _stream(stream))
    _check(rc, "pa_decode")


def pa_decode_ex(out, q, k_cache, v_cache, block_table, seq_lens, scale: float, num_kv_heads: int,
                 k_scale=None, v_scale=None, partition_size: int = 0, workspace=None, device_error=None,
                 stream=None) -> None:
    """pa_decode with FP8 scales, explicit partition size (0 heuristic, -1 unsplit), caller workspace
    (a zero-filled uint8 CUDA tensor, see pa_decode_workspace_size) and device error word (int32)."""
    args = (desc(out), desc(q), desc(k_cache), desc(v_cache), desc(block_table), desc(seq_lens))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().pa_decode_ex(*[ctypes.byref(a) for a in args], float(scale), int(num_kv_heads), _ptr(k_scale),
                            _ptr(v_scale), int(partition_size), _ptr(workspace), ws_bytes, _ptr(device_error),
                            _stream(stream))
    _check(rc, "pa_decode_ex")


def pa_decode_noalloc(out, q, k_cache, v_cache, block_table, seq_lens, scale: float, num_kv_heads: int,
                      k_scale=None, v_scale=None, partition_size: int = 0, device_error=None, stream=None) -> None:
    """pa_decode_ex without a workspace argument: for callers that cannot allocate device memory
    where they run decode.  Split-KV scratch comes from a fixed 32 MiB buffer inside the library,
    shared by all calls on a device (calls that overlap on the GPU race on it); a problem needing
    more than that raises PAError(PA_ERR_WORKSPACE)."""
    args = (desc(out), desc(q), desc(k_cache), desc(v_cache), desc(block_table), desc(seq_lens))
    rc = lib().pa_decode_noalloc(*[ctypes.byref(a) for a in args], float(scale), int(num_kv_heads), _ptr(k_scale),
                                 _ptr(v_scale), int(partition_size), _ptr(device_error), _stream(stream))
    _check(rc, "pa_decode_noalloc")


def pa_decode_plan(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, kv_dtype_code,
                   sm_count=0, partition_size=0):
    """(partition tokens or 0 for unsplit, partitions of the longest sequence) -- host only."""
    P, n = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().pa_decode_plan(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, kv_dtype_code,
                              sm_count, partition_size, ctypes.byref(P), ctypes.byref(n))
    _check(rc, "pa_decode_plan")
    return P.value, n.value


def pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq, partition_size) -> int:
    """Bytes of split-KV workspace; zero-fill it once before first use (torch.zeros)."""
    return int(lib().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, max_blocks_per_seq,
                                              partition_size))


def pa_check_device_error(device_error, stream=None):
    """(status, bits); synchronises the stream and resets the word."""
    bits = ctypes.c_int(0)
    rc = lib().pa_check_device_error(_ptr(device_error), ctypes.byref(bits), _stream(stream))
    return rc, bits.value


def pa_status_string(status: int) -> str:
    return status_string(status)


def pa_profile_enable(on: bool = True) -> None:
    _check(lib().pa_profile_enable(1 if on else 0), "pa_profile_enable")


def pa_profile_read(kind: int):
    """(total device ms, launches) for kind PA_KERNEL_WRITE / PA_KERNEL_DECODE since the last read."""
    ms, n = ctypes.c_double(0), ctypes.c_longlong(0)
    _check(lib().pa_profile_read(int(kind), ctypes.byref(ms), ctypes.byref(n)), "pa_profile_read")
    return ms.value, n.value


class BlockManager:
    """The C block manager (pa_bm_*): free list, per-sequence block tables, reference-counted
    prefix sharing with copy on write.  Host only."""

    def __init__(self, num_blocks: int, max_seqs: int, max_blocks_per_seq: int):
        self._m = lib().pa_bm_create(int(num_blocks), int(max_seqs), int(max_blocks_per_seq))
        if not self._m:
            raise PAError(-1, "pa_bm_create")
        self.max_blocks_per_seq = int(max_blocks_per_seq)

    def close(self):
        if self._m:
            lib().pa_bm_destroy(self._m)
            self._m = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return lib().pa_bm_num_free(self._m)

    def refs(self, block: int) -> int:
        return lib().pa_bm_block_refs(self._m, int(block))

    def seq_len(self, seq: int) -> int:
        return lib().pa_bm_seq_len(self._m, int(seq))

    def append(self, seq: int, n_tokens: int):
        """(slots int64 [n_tokens], copy pair (src, dst) or None)."""
        import numpy as np
        slots = np.zeros(max(int(n_tokens), 1), dtype=np.int64)
        pair = np.zeros(2, dtype=np.int64)
        nc = ctypes.c_int(0)
        i64p = ctypes.POINTER(ctypes.c_int64)
        rc = lib().pa_bm_append(self._m, int(seq), int(n_tokens), slots.ctypes.data_as(i64p),
                                pair.ctypes.data_as(i64p), ctypes.byref(nc))
        _check(rc, "pa_bm_append")
        return slots[:int(n_tokens)], ((int(pair[0]), int(pair[1])) if nc.value else None)

    def fork(self, src: int, dst: int) -> None:
        _check(lib().pa_bm_fork(self._m, int(src), int(dst)), "pa_bm_fork")

    def free(self, seq: int) -> None:
        _check(lib().pa_bm_free(self._m, int(seq)), "pa_bm_free")

    def export(self, seqs, row_stride: int | None = None):
        """(block_table int32 [n, row_stride], seq_lens int32 [n]) as numpy arrays."""
        import numpy as np
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        rs = self.max_blocks_per_seq if row_stride is None else int(row_stride)
        bt = np.zeros((len(seqs), rs), dtype=np.int32)
        sl = np.zeros(len(seqs), dtype=np.int32)
        i32p = ctypes.POINTER(ctypes.c_int32)
        rc = lib().pa_bm_export(self._m, seqs.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), len(seqs), rs,
                                bt.ctypes.data_as(i32p), sl.ctypes.data_as(i32p))
        _check(rc, "pa_bm_export")
        return bt, sl


def pa_copy_blocks(k_cache, v_cache, block_pairs, device_error=None, stream=None) -> None:
    """Copy whole cache blocks: for each row (src, dst) of block_pairs (int64 [n, 2] on the
    device), block src of k_cache / v_cache is copied to block dst."""
    args = (desc(k_cache), desc(v_cache), desc(block_pairs))
    rc = lib().pa_copy_blocks(*[ctypes.byref(a) for a in args], _ptr(device_error), _stream(stream))
    _check(rc, "pa_copy_blocks")
