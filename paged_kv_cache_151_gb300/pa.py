"""Python binding of the C ABI in ``include/pa.h`` (argument marshalling only).

Each function takes torch tensors that live on the current CUDA device, reads
their pointers, sizes and strides, and calls the function of the same name in
``libpa.so`` on ``torch.cuda.current_stream()``.  Every step of the path runs
in the library's kernels; this module computes nothing.  A non-zero status
raises ``PAError``.  If the library is missing it is built from source (nvcc);
if that is impossible the call fails loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

PA_F32, PA_BF16, PA_F16, PA_E4M3 = 0, 1, 2, 3
_DTYPE = {torch.float32: PA_F32, torch.bfloat16: PA_BF16, torch.float16: PA_F16}

PA_DEVERR_BLOCK_ID = 0x1
PA_DEVERR_SEQ_LEN = 0x2
PA_DEVERR_SLOT = 0x4
PA_DEVERR_TIMEOUT = 0x8


class PAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {pa_status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load ``libpa.so`` (building it first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            path = _build.build()
        lib = ctypes.CDLL(path)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                ctypes.c_float, ctypes.c_size_t)
        lib.pa_abi_version.restype = ctypes.c_int
        lib.pa_abi_version.argtypes = []
        lib.pa_test_stall_next_decode.restype = ctypes.c_int
        lib.pa_test_stall_next_decode.argtypes = []
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_status_string.argtypes = [ctypes.c_int]
        lib.pa_reshape_and_cache.restype = ctypes.c_int
        lib.pa_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i32, i32, i64, i64, i64,
                                             i32, i32, P]
        dec = [P, P, P, P, P, P, i32, i32, i32, i32, i64, i32, i32, i64, f32, i32]
        lib.pa_decode.restype = ctypes.c_int
        lib.pa_decode.argtypes = dec + [P]
        lib.pa_decode_split.restype = ctypes.c_int
        lib.pa_decode_split.argtypes = dec + [i32, P]
        lib.pa_decode_partitioned_workspace_size.restype = sz
        lib.pa_decode_partitioned_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.pa_decode_partitioned.restype = ctypes.c_int
        lib.pa_decode_partitioned.argtypes = dec + [i32, i32, P, sz, P]
        lib.pa_decode_partitioned_noalloc.restype = ctypes.c_int
        lib.pa_decode_partitioned_noalloc.argtypes = dec + [i32, i32, P]
        lib.pa_decode_cascade_workspace_size.restype = sz
        lib.pa_decode_cascade_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.pa_decode_cascade.restype = ctypes.c_int
        lib.pa_decode_cascade.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i64, i32,
                                          i32, i64, f32, i32, P, sz, P]
        lib.pa_decode_multi.restype = ctypes.c_int
        lib.pa_decode_multi.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                        i64, i32, i32, i64, f32, i32, P]
        lib.pa_reshape_and_cache_fp8.restype = ctypes.c_int
        lib.pa_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i64, i64,
                                                 i64, i32, i32, P]
        dec8 = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i64, i32, i32, i64, f32, i32]
        lib.pa_decode_fp8.restype = ctypes.c_int
        lib.pa_decode_fp8.argtypes = dec8 + [P]
        lib.pa_decode_partitioned_fp8.restype = ctypes.c_int
        lib.pa_decode_partitioned_fp8.argtypes = dec8 + [i32, i32, P, sz, P]
        lib.pa_copy_blocks.restype = ctypes.c_int
        lib.pa_copy_blocks.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32, P, i64, i64, i64,
                                       P]
        lib.pa_device_error.restype = ctypes.c_int
        lib.pa_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        _lib = lib
        return lib


def pa_status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def pa_abi_version() -> int:
    return int(load().pa_abi_version())


def _check(fn: str, rc: int):
    if rc != 0:
        raise PAError(fn, rc)


def _dev(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is not on the current device")


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _cache_dims(k_cache: torch.Tensor, v_cache: torch.Tensor):
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("caches must both be [num_blocks, num_kv_heads, block_size, head_dim]")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    if k_cache.dtype != v_cache.dtype or k_cache.dtype not in _DTYPE:
        raise ValueError("caches must share a dtype in {float32, bfloat16, float16}")
    return k_cache.shape


def pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """Write k[t], v[t] ([T, H_kv, D], heads contiguous) into their slots."""
    for n, t in (("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("slot_mapping", slot_mapping)):
        _dev(t, n)
    N, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    if k.dim() != 3 or k.shape != v.shape or tuple(k.shape[1:]) != (Hkv, D):
        raise ValueError("k and v must be [num_tokens, num_kv_heads, head_dim]")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype:
        raise ValueError("k, v and the caches must share a dtype")
    if k.stride(2) != 1 or k.stride(1) != D or v.stride(2) != 1 or v.stride(1) != D:
        raise ValueError("k and v must have contiguous heads")
    if slot_mapping.dtype != torch.int64 or slot_mapping.dim() != 1 or \
            slot_mapping.shape[0] != k.shape[0] or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 [num_tokens]")
    rc = load().pa_reshape_and_cache(
        k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        slot_mapping.data_ptr(), k.shape[0], Hkv, D, k.stride(0), v.stride(0), N, bs,
        _DTYPE[k.dtype], _stream(stream))
    _check("pa_reshape_and_cache", rc)


def _decode_args(out, q, k_cache, v_cache, block_tables, seq_lens):
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("seq_lens", seq_lens)):
        _dev(t, n)
    N, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    if q.dim() != 3 or q.shape[2] != D or q.stride(2) != 1 or q.stride(1) != D:
        raise ValueError("q must be [num_seqs, num_heads, head_dim] with contiguous heads")
    if out.shape != q.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like q")
    if q.dtype != k_cache.dtype or out.dtype != k_cache.dtype:
        raise ValueError("q, out and the caches must share a dtype")
    B, H = q.shape[0], q.shape[1]
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or \
            block_tables.shape[0] != B or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous int32 [num_seqs, max_blocks]")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,) or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 [num_seqs]")
    return [out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
            block_tables.data_ptr(), seq_lens.data_ptr(), B, H, Hkv, D, N, bs,
            block_tables.shape[1], q.stride(0)]


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale, num_kv_heads,
              stream=None):
    """Decode-step paged attention into ``out`` ([B, H_q, D])."""
    args = _decode_args(out, q, k_cache, v_cache, block_tables, seq_lens)
    if num_kv_heads != k_cache.shape[1]:
        raise ValueError("num_kv_heads does not match the cache")
    rc = load().pa_decode(*args, float(scale), _DTYPE[q.dtype], _stream(stream))
    _check("pa_decode", rc)


def pa_decode_split(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                    num_kv_heads, splits, stream=None):
    """pa_decode with an explicit cluster split (1, 2, 4, 8; 0 = automatic)."""
    args = _decode_args(out, q, k_cache, v_cache, block_tables, seq_lens)
    if num_kv_heads != k_cache.shape[1]:
        raise ValueError("num_kv_heads does not match the cache")
    rc = load().pa_decode_split(*args, float(scale), _DTYPE[q.dtype], int(splits),
                                _stream(stream))
    _check("pa_decode_split", rc)


def pa_decode_partitioned_workspace_size(num_seqs, num_heads, head_dim, max_seq_len,
                                         partition_size) -> int:
    return int(load().pa_decode_partitioned_workspace_size(
        int(num_seqs), int(num_heads), int(head_dim), int(max_seq_len),
        int(partition_size)))


def pa_decode_partitioned(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                          num_kv_heads, partition_size, max_seq_len, workspace,
                          stream=None):
    """Split-KV decode; ``workspace`` is a CUDA uint8 tensor of at least
    ``pa_decode_partitioned_workspace_size(...)`` bytes, 256-byte aligned."""
    args = _decode_args(out, q, k_cache, v_cache, block_tables, seq_lens)
    if num_kv_heads != k_cache.shape[1]:
        raise ValueError("num_kv_heads does not match the cache")
    _dev(workspace, "workspace")
    nbytes = workspace.numel() * workspace.element_size()
    rc = load().pa_decode_partitioned(*args, float(scale), _DTYPE[q.dtype],
                                      int(partition_size), int(max_seq_len),
                                      workspace.data_ptr(), nbytes, _stream(stream))
    _check("pa_decode_partitioned", rc)


def pa_decode_cascade_workspace_size(num_seqs, num_heads, head_dim, num_prefix_blocks,
                                     max_blocks_per_seq) -> int:
    return int(load().pa_decode_cascade_workspace_size(
        int(num_seqs), int(num_heads), int(head_dim), int(num_prefix_blocks),
        int(max_blocks_per_seq)))


def pa_decode_cascade(out, q, k_cache, v_cache, prefix_blocks, block_tables, seq_lens, scale,
                      num_kv_heads, workspace, stream=None):
    """Decode for sequences that all begin with the physical blocks
    ``prefix_blocks`` (int32 [P], on the device): sequence s attends over the
    16 * P prefix tokens, then seq_lens[s] tokens of its own in
    block_tables[s].  ``workspace``: a CUDA uint8 tensor of at least
    ``pa_decode_cascade_workspace_size(...)`` bytes, 256-byte aligned."""
    args = _decode_args(out, q, k_cache, v_cache, block_tables, seq_lens)
    if num_kv_heads != k_cache.shape[1]:
        raise ValueError("num_kv_heads does not match the cache")
    _dev(prefix_blocks, "prefix_blocks")
    if prefix_blocks.dtype != torch.int32 or prefix_blocks.dim() != 1 or \
            not prefix_blocks.is_contiguous():
        raise ValueError("prefix_blocks must be a contiguous int32 [num_prefix_blocks]")
    _dev(workspace, "workspace")
    nbytes = workspace.numel() * workspace.element_size()
    out_p, q_p, kc, vc, bt, sl = args[:6]
    rest = args[6:]                                # B, H, Hkv, D, N, bs, max_blocks, q stride
    rc = load().pa_decode_cascade(out_p, q_p, kc, vc, prefix_blocks.data_ptr(),
                                  prefix_blocks.shape[0], bt, sl, *rest, float(scale),
                                  _DTYPE[q.dtype], workspace.data_ptr(), nbytes,
                                  _stream(stream))
    _check("pa_decode_cascade", rc)


# Bytes of the workspace built into the library for the call below.
PA_NOALLOC_SCRATCH_BYTES = 32 << 20


def pa_decode_partitioned_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                                  num_kv_heads, partition_size, max_seq_len, stream=None):
    """Split-KV decode for callers that cannot allocate device memory: the
    partition workspace is the library's built-in array of
    PA_NOALLOC_SCRATCH_BYTES (shared by every call on the device, so calls
    that may overlap on the GPU must be serialised).  The first call on a
    device looks up that array; make it before any stream capture."""
    args = _decode_args(out, q, k_cache, v_cache, block_tables, seq_lens)
    if num_kv_heads != k_cache.shape[1]:
        raise ValueError("num_kv_heads does not match the cache")
    rc = load().pa_decode_partitioned_noalloc(*args, float(scale), _DTYPE[q.dtype],
                                              int(partition_size), int(max_seq_len),
                                              _stream(stream))
    _check("pa_decode_partitioned_noalloc", rc)


def pa_decode_multi(out, q, k_cache, v_cache, block_tables, seq_lens, query_start,
                    max_query_len, scale, num_kv_heads, stream=None):
    """Paged attention of several new tokens per sequence: q and out are
    [T, H_q, D] with the rows of sequence s at query_start[s] ..
    query_start[s+1]-1 (int32 [B+1]); row i of a sequence with n rows sees
    positions 0 .. seq_lens[s] - n + i of its cache."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("seq_lens", seq_lens),
                 ("query_start", query_start)):
        _dev(t, n)
    N, Hkv, bs, D = _cache_dims(k_cache, v_cache)
    if num_kv_heads != Hkv:
        raise ValueError("num_kv_heads does not match the cache")
    if q.dim() != 3 or q.shape[2] != D or q.stride(2) != 1 or q.stride(1) != D:
        raise ValueError("q must be [num_rows, num_heads, head_dim] with contiguous heads")
    if out.shape != q.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped like q")
    if q.dtype != k_cache.dtype or out.dtype != k_cache.dtype:
        raise ValueError("q, out and the caches must share a dtype")
    if seq_lens.dtype != torch.int32 or seq_lens.dim() != 1 or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 [num_seqs]")
    B = seq_lens.shape[0]
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or \
            block_tables.shape[0] != B or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous int32 [num_seqs, max_blocks]")
    if query_start.dtype != torch.int32 or query_start.shape != (B + 1,) or \
            not query_start.is_contiguous():
        raise ValueError("query_start must be a contiguous int32 [num_seqs + 1]")
    rc = load().pa_decode_multi(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), seq_lens.data_ptr(), query_start.data_ptr(), B,
        q.shape[0], int(max_query_len), q.shape[1], Hkv, D, N, bs, block_tables.shape[1],
        q.stride(0), float(scale), _DTYPE[q.dtype], _stream(stream))
    _check("pa_decode_multi", rc)


def pa_copy_blocks(caches, block_mapping, stream=None):
    """Copy-on-write block copies: for every (src, dst) row of ``block_mapping``
    (CUDA int64 [P, 2]) copy block src to block dst in every tensor of
    ``caches`` (contiguous CUDA tensors [num_blocks, ...] of one shape, e.g. K
    and V of every layer)."""
    caches = list(caches)
    _dev(block_mapping, "block_mapping")
    if block_mapping.dtype != torch.int64 or block_mapping.dim() != 2 or \
            block_mapping.shape[1] != 2 or not block_mapping.is_contiguous():
        raise ValueError("block_mapping must be a contiguous int64 [num_pairs, 2]")
    if not caches:
        return
    shape = caches[0].shape
    nbytes = caches[0].numel() * caches[0].element_size()
    for i, c in enumerate(caches):
        _dev(c, f"caches[{i}]")
        if c.shape != shape or not c.is_contiguous() or \
                c.numel() * c.element_size() != nbytes:
            raise ValueError("caches must be contiguous tensors of one shape and size")
    num_blocks = shape[0]
    block_bytes = nbytes // max(num_blocks, 1)
    ptrs = (ctypes.c_void_p * len(caches))(*[c.data_ptr() for c in caches])
    rc = load().pa_copy_blocks(ptrs, len(caches), block_mapping.data_ptr(),
                               block_mapping.shape[0], num_blocks, block_bytes,
                               _stream(stream))
    _check("pa_copy_blocks", rc)


# ---- FP8 (E4M3) cache ------------------------------------------------------

_FP8_TYPES = tuple(t for t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) if t)


def _fp8_cache_dims(k_cache, v_cache, k_scale, v_scale):
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_scale", k_scale),
                 ("v_scale", v_scale)):
        _dev(t, n)
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("caches must both be [num_blocks, num_kv_heads, block_size, head_dim]")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    if k_cache.dtype not in _FP8_TYPES or v_cache.dtype not in _FP8_TYPES:
        raise ValueError("FP8 caches hold E4M3 codes (uint8 or float8_e4m3fn tensors)")
    Hkv = k_cache.shape[1]
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t.dtype != torch.float32 or t.shape != (Hkv,) or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float32 [num_kv_heads]")
    return k_cache.shape


def pa_reshape_and_cache_fp8(k, v, k_cache, v_cache, k_scale, v_scale, slot_mapping,
                             stream=None):
    """Write k[t], v[t] ([T, H_kv, D] in f32/bf16/f16) into E4M3 caches as
    E4M3(x / scale[j])."""
    for n, t in (("k", k), ("v", v), ("slot_mapping", slot_mapping)):
        _dev(t, n)
    N, Hkv, bs, D = _fp8_cache_dims(k_cache, v_cache, k_scale, v_scale)
    if k.dim() != 3 or k.shape != v.shape or tuple(k.shape[1:]) != (Hkv, D):
        raise ValueError("k and v must be [num_tokens, num_kv_heads, head_dim]")
    if k.dtype not in _DTYPE or v.dtype != k.dtype:
        raise ValueError("k and v must share a dtype in {float32, bfloat16, float16}")
    if k.stride(2) != 1 or k.stride(1) != D or v.stride(2) != 1 or v.stride(1) != D:
        raise ValueError("k and v must have contiguous heads")
    if slot_mapping.dtype != torch.int64 or slot_mapping.dim() != 1 or \
            slot_mapping.shape[0] != k.shape[0] or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 [num_tokens]")
    rc = load().pa_reshape_and_cache_fp8(
        k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        k_scale.data_ptr(), v_scale.data_ptr(), slot_mapping.data_ptr(), k.shape[0], Hkv, D,
        k.stride(0), v.stride(0), N, bs, _DTYPE[k.dtype], _stream(stream))
    _check("pa_reshape_and_cache_fp8", rc)


def _decode_fp8_args(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens):
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables),
                 ("seq_lens", seq_lens)):
        _dev(t, n)
    N, Hkv, bs, D = _fp8_cache_dims(k_cache, v_cache, k_scale, v_scale)
    if q.dim() != 3 or q.shape[2] != D or q.stride(2) != 1 or q.stride(1) != D:
        raise ValueError("q must be [num_seqs, num_heads, head_dim] with contiguous heads")
    if out.shape != q.shape or not out.is_contiguous() or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous tensor shaped and typed like q")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q must be bfloat16 or float16")
    B, H = q.shape[0], q.shape[1]
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or \
            block_tables.shape[0] != B or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous int32 [num_seqs, max_blocks]")
    if seq_lens.dtype != torch.int32 or seq_lens.shape != (B,) or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 [num_seqs]")
    return [out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
            k_scale.data_ptr(), v_scale.data_ptr(), block_tables.data_ptr(),
            seq_lens.data_ptr(), B, H, Hkv, D, N, bs, block_tables.shape[1], q.stride(0)]


def pa_decode_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens,
                  scale, num_kv_heads, stream=None):
    """Decode-step paged attention over E4M3 caches into ``out``."""
    args = _decode_fp8_args(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                            seq_lens)
    if num_kv_heads != k_cache.shape[1]:
        raise ValueError("num_kv_heads does not match the cache")
    rc = load().pa_decode_fp8(*args, float(scale), _DTYPE[q.dtype], _stream(stream))
    _check("pa_decode_fp8", rc)


def pa_decode_partitioned_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                              seq_lens, scale, num_kv_heads, partition_size, max_seq_len,
                              workspace, stream=None):
    """Split-KV decode over E4M3 caches (workspace as pa_decode_partitioned)."""
    args = _decode_fp8_args(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                            seq_lens)
    if num_kv_heads != k_cache.shape[1]:
        raise ValueError("num_kv_heads does not match the cache")
    _dev(workspace, "workspace")
    nbytes = workspace.numel() * workspace.element_size()
    rc = load().pa_decode_partitioned_fp8(*args, float(scale), _DTYPE[q.dtype],
                                          int(partition_size), int(max_seq_len),
                                          workspace.data_ptr(), nbytes, _stream(stream))
    _check("pa_decode_partitioned_fp8", rc)


def workspace_views(workspace, num_seqs, num_heads, head_dim, max_seq_len, partition_size):
    """(o_part, m_part, l_part) fp32 views of a partitioned-decode workspace,
    following the layout documented in include/pa.h."""
    P = max(1, -(-int(max_seq_len) // int(partition_size)))
    rows = num_seqs * num_heads * P

    def up(x):
        return (x + 255) // 256 * 256
    off_m = up(rows * head_dim * 4)
    off_l = off_m + up(rows * 4)
    f = workspace.view(torch.uint8)
    o = f[:rows * head_dim * 4].view(torch.float32).view(num_seqs, num_heads, P, head_dim)
    m = f[off_m:off_m + rows * 4].view(torch.float32).view(num_seqs, num_heads, P)
    l = f[off_l:off_l + rows * 4].view(torch.float32).view(num_seqs, num_heads, P)
    return o, m, l


def pa_test_stall_next_decode() -> None:
    """Test hook: in the next decode call each warp's first copy never completes,
    so its bounded wait runs out and the call sets PA_DEVERR_TIMEOUT."""
    _check("pa_test_stall_next_decode", load().pa_test_stall_next_decode())


def pa_device_error(clear: bool = True) -> int:
    """Sticky device error bits (PA_DEVERR_*); synchronises the device."""
    flags = ctypes.c_uint32(0)
    _check("pa_device_error", load().pa_device_error(ctypes.byref(flags), int(clear)))
    return int(flags.value)


__all__ = [
    "PAError", "load", "library_path", "pa_status_string", "pa_abi_version",
    "pa_test_stall_next_decode",
    "pa_reshape_and_cache", "pa_decode", "pa_decode_split",
    "pa_decode_partitioned_workspace_size", "pa_decode_partitioned", "pa_decode_multi",
    "pa_decode_partitioned_noalloc", "PA_NOALLOC_SCRATCH_BYTES",
    "pa_decode_cascade", "pa_decode_cascade_workspace_size",
    "pa_reshape_and_cache_fp8", "pa_decode_fp8", "pa_decode_partitioned_fp8",
    "pa_copy_blocks",
    "pa_device_error", "workspace_views",
    "PA_DEVERR_BLOCK_ID", "PA_DEVERR_SEQ_LEN", "PA_DEVERR_SLOT", "PA_DEVERR_TIMEOUT",
]
