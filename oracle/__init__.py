"""fp64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``pa_ref.c`` (plain C, built
with gcc) and shares no code with the CUDA library: it never imports the
product package and the product never imports it.

Every function takes host data (numpy arrays or CPU torch tensors) and returns
fp64 numpy arrays.  The arithmetic is documented in ``pa_ref.c``:

* ``reshape_and_cache``  -- byte copy of each new K/V row into its slot
  ("vLLM: Architecture, PagedAttention & Internals", *The forward step in
  detail*).
* ``decode`` / ``decode_one`` -- gather through the block table, then
  textbook softmax attention in fp64 (same page, *PagedAttention in one
  paragraph*).
* ``decode_multi`` -- several new query tokens per sequence, each attending
  causally to the cache up to its own position (chunked prefill and
  speculative verification over the paged cache).
* ``partition_stats`` / ``lse_merge`` -- split-KV partition statistics and
  their log-sum-exp merge.
* ``kv_bytes_per_token`` / ``bytes_per_block`` / ``blocks_for_tokens`` --
  the pages' KV sizing arithmetic.
* ``copy_blocks`` -- the block copies of copy-on-write ("vLLM: Architecture,
  PagedAttention & Internals", *Copy-on-write for shared blocks*).
* ``e4m3_encode`` / ``e4m3_decode`` / ``reshape_and_cache_fp8`` and the
  ``kv_scales=`` form of ``decode`` / ``decode_one`` -- the FP8 (E4M3) KV
  cache with one scale per KV head for K and for V.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpa_ref.so")
_lock = threading.Lock()
_lib = None

REF_DTYPE = {"f32": 0, "bf16": 1, "f16": 2}


def build(force: bool = False) -> str:
    """Compile pa_ref.c into oracle/_build/libpa_ref.so (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load a build of pa_ref.c from ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.pa_ref_kv_bytes_per_token.restype = i64
    lib.pa_ref_kv_bytes_per_token.argtypes = [i64, i64, i64, i64]
    lib.pa_ref_bytes_per_block.restype = i64
    lib.pa_ref_bytes_per_block.argtypes = [i64, i64, i64, i64, i64]
    lib.pa_ref_blocks_for_tokens.restype = i64
    lib.pa_ref_blocks_for_tokens.argtypes = [i64, i64]
    lib.pa_ref_reshape_and_cache.restype = i64
    lib.pa_ref_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i32, i32,
                                             i64, i64, i32, i64, i32]
    common = [P, P, P, P, P, i64, i32, i32, i32, i32, i64, i64, i64, i64, f32, i32]
    lib.pa_ref_decode.restype = ctypes.c_int
    lib.pa_ref_decode.argtypes = [P] + common + [i32]
    lib.pa_ref_decode_one.restype = ctypes.c_int
    lib.pa_ref_decode_one.argtypes = [P, P, i64, i32] + common
    lib.pa_ref_partition_stats.restype = i64
    lib.pa_ref_partition_stats.argtypes = [P, P, P, i64, i32, i32] + common
    lib.pa_ref_decode_multi.restype = ctypes.c_int
    lib.pa_ref_decode_multi.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i32, i32, i64,
                                        i64, i64, f32, i32]
    lib.pa_ref_e4m3_to_double.restype = ctypes.c_double
    lib.pa_ref_e4m3_to_double.argtypes = [i32]
    lib.pa_ref_e4m3_from_float.restype = i32
    lib.pa_ref_e4m3_from_float.argtypes = [f32]
    lib.pa_ref_reshape_and_cache_fp8.restype = i64
    lib.pa_ref_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, i64, i32, i32, i64, i64,
                                                 i32, i64, i32, P, P]
    lib.pa_ref_decode_fp8.restype = ctypes.c_int
    lib.pa_ref_decode_fp8.argtypes = [P] + common + [P, P, i32]
    lib.pa_ref_decode_one_fp8.restype = ctypes.c_int
    lib.pa_ref_decode_one_fp8.argtypes = [P, P, i64, i32] + common + [P, P]
    lib.pa_ref_copy_blocks.restype = i64
    lib.pa_ref_copy_blocks.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32, P, i64, i64, i64]
    lib.pa_ref_lse_merge.restype = None
    lib.pa_ref_lse_merge.argtypes = [P, P, P, P, i64, i32]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
        return _lib


def build_variant(src_text: str, out_dir: str) -> str:
    """Compile an edited copy of the oracle source (used by the tests that
    check that the pins catch planted mistakes).  Returns the library path."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "variant.c")
    lib = os.path.join(out_dir, "libvariant.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                    "-fno-fast-math", "-ffp-contract=off", "-pthread", src,
                    "-o", lib, "-lm"], check=True)
    return lib


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


_override = threading.local()


def _active():
    lib = getattr(_override, "lib", None)
    return lib if lib is not None else _load()


class use_library:
    """Context manager: route this thread's oracle calls to another build."""

    def __init__(self, path: str):
        self.lib = bind(path)

    def __enter__(self):
        self.prev = getattr(_override, "lib", None)
        _override.lib = self.lib
        return self

    def __exit__(self, *exc):
        _override.lib = self.prev
        return False


# ---- host-buffer helpers --------------------------------------------------

def _host(x, np_dtype=None) -> np.ndarray:
    """A C-contiguous numpy view (or copy) of a numpy array / CPU tensor.
    bf16 and f16 tensors are viewed as uint16 bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach()
            if x.device.type != "cpu":
                raise ValueError("oracle takes host tensors")
            if x.dtype in (torch.bfloat16, torch.float16):
                x = x.contiguous().view(torch.int16).numpy().view(np.uint16)
            elif x.dtype in (getattr(torch, "float8_e4m3fn", None), torch.uint8):
                x = x.contiguous().view(torch.uint8).numpy()
            else:
                x = x.contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if np_dtype is not None and x.dtype != np_dtype:
        x = x.astype(np_dtype)
    return x


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def kv_bytes_per_token(num_layers, num_kv_heads, head_dim, dtype_bytes) -> int:
    return int(_active().pa_ref_kv_bytes_per_token(num_layers, num_kv_heads,
                                                 head_dim, dtype_bytes))


def bytes_per_block(block_size, num_layers, num_kv_heads, head_dim, dtype_bytes) -> int:
    return int(_active().pa_ref_bytes_per_block(block_size, num_layers,
                                              num_kv_heads, head_dim, dtype_bytes))


def blocks_for_tokens(n_tokens, block_size) -> int:
    return int(_active().pa_ref_blocks_for_tokens(n_tokens, block_size))


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, dtype: str):
    """Return (k_cache', v_cache', n_bad) after writing the new rows.
    ``k``/``v``: [T, H_kv, D]; caches [N, H_kv, bs, D] (copied, not modified)."""
    lib = _active()
    k = _host(k); v = _host(v)
    kc = _host(k_cache).copy(); vc = _host(v_cache).copy()
    sm = _host(slot_mapping, np.int64)
    T, Hkv, D = k.shape
    N, _, bs, _ = kc.shape
    bad = lib.pa_ref_reshape_and_cache(_p(k), _p(v), _p(kc), _p(vc), _p(sm), T,
                                       Hkv, D, Hkv * D, Hkv * D, bs, N,
                                       REF_DTYPE[dtype])
    return kc, vc, int(bad)


def copy_blocks(caches, block_mapping):
    """Copy-on-write block copies: return (copies of the caches, n_bad).
    ``caches``: arrays/CPU tensors [num_blocks, ...] of one shape and dtype
    (e.g. K and V of every layer); ``block_mapping``: int64 [P, 2] (src, dst),
    applied in order."""
    hs = [_host(c).copy() for c in caches]
    if not hs:
        return [], 0
    n = hs[0].shape[0]
    for h in hs:
        if h.shape != hs[0].shape or h.dtype != hs[0].dtype:
            raise ValueError("caches must share shape and dtype")
    bb = hs[0].nbytes // max(n, 1)
    m = _host(block_mapping, np.int64).reshape(-1, 2)
    ptrs = (ctypes.c_void_p * len(hs))(*[h.ctypes.data for h in hs])
    bad = _active().pa_ref_copy_blocks(ptrs, len(hs), _p(np.ascontiguousarray(m)),
                                       m.shape[0], n, bb)
    return hs, int(bad)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of binary32 values: nearest, ties to even,
    saturating at +-448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float32)
    f = _active().pa_ref_e4m3_from_float
    return np.array([f(float(v)) for v in x.reshape(-1)], dtype=np.uint8).reshape(x.shape)


def e4m3_decode(codes) -> np.ndarray:
    """Values (fp64) of E4M3 codes."""
    c = np.asarray(codes, dtype=np.uint8)
    f = _active().pa_ref_e4m3_to_double
    return np.array([f(int(v)) for v in c.reshape(-1)], dtype=np.float64).reshape(c.shape)


def reshape_and_cache_fp8(k, v, k_cache, v_cache, slot_mapping, dtype: str, k_scale,
                          v_scale):
    """FP8 cache write: return (k_cache', v_cache', n_bad) with the new rows
    stored as E4M3(x / scale[j]).  ``k``/``v``: [T, H_kv, D] in ``dtype``;
    caches: E4M3 codes [N, H_kv, bs, D] (copied, not modified); scales [H_kv]."""
    lib = _active()
    k = _host(k); v = _host(v)
    kc = _host(k_cache).copy(); vc = _host(v_cache).copy()
    sm = _host(slot_mapping, np.int64)
    ks = _host(k_scale, np.float32); vs = _host(v_scale, np.float32)
    T, Hkv, D = k.shape
    N, _, bs, _ = kc.shape
    if ks.shape != (Hkv,) or vs.shape != (Hkv,):
        raise ValueError("one K and one V scale per KV head")
    bad = lib.pa_ref_reshape_and_cache_fp8(_p(k), _p(v), _p(kc), _p(vc), _p(sm), T, Hkv,
                                           D, Hkv * D, Hkv * D, bs, N, REF_DTYPE[dtype],
                                           _p(ks), _p(vs))
    return kc, vc, int(bad)


class _Problem:
    """Marshalled arguments shared by the decode entry points.  With
    ``kv_scales=(k_scale, v_scale)`` the caches hold E4M3 codes and ``dtype``
    is the type of q."""

    def __init__(self, q, k_cache, v_cache, block_tables, seq_lens, scale,
                 num_kv_heads, dtype, kv_scales=None):
        self.q = _host(q)
        self.kc = _host(k_cache)
        self.vc = _host(v_cache)
        self.bt = _host(block_tables, np.int32)
        self.sl = _host(seq_lens, np.int32)
        self.B, self.H, self.D = self.q.shape
        self.N, kvh, self.bs, _ = self.kc.shape
        if kvh != num_kv_heads:
            raise ValueError("num_kv_heads does not match the cache")
        self.Hkv = num_kv_heads
        self.max_blocks = self.bt.shape[1]
        self.scale = float(scale)
        self.dtype = REF_DTYPE[dtype]
        self.fp8 = kv_scales is not None
        if self.fp8:
            self.ks = _host(kv_scales[0], np.float32)
            self.vs = _host(kv_scales[1], np.float32)
            if self.ks.shape != (kvh,) or self.vs.shape != (kvh,):
                raise ValueError("one K and one V scale per KV head")
            if self.kc.dtype != np.uint8:
                raise ValueError("FP8 caches hold uint8 E4M3 codes")

    def scales(self):
        return [_p(self.ks), _p(self.vs)]

    def common(self):
        return [_p(self.q), _p(self.kc), _p(self.vc), _p(self.bt), _p(self.sl),
                self.B, self.H, self.Hkv, self.D, self.bs, self.N,
                self.max_blocks, self.H * self.D, self.D, self.scale, self.dtype]


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, num_kv_heads,
           dtype: str, nthreads: int = 1, kv_scales=None) -> np.ndarray:
    """fp64 decode attention for every (sequence, query head): [B, H_q, D].
    ``kv_scales=(k_scale, v_scale)``: E4M3 caches with per-KV-head scales."""
    pr = _Problem(q, k_cache, v_cache, block_tables, seq_lens, scale,
                  num_kv_heads, dtype, kv_scales)
    out = np.zeros((pr.B, pr.H, pr.D), dtype=np.float64)
    if pr.fp8:
        rc = _active().pa_ref_decode_fp8(_p(out), *pr.common(), *pr.scales(), int(nthreads))
    else:
        rc = _active().pa_ref_decode(_p(out), *pr.common(), int(nthreads))
    if rc:
        raise ValueError("oracle decode: invalid input (block id or seq_len out of range)")
    return out


def decode_one(s, h, q, k_cache, v_cache, block_tables, seq_lens, scale,
               num_kv_heads, dtype: str, problem: _Problem | None = None):
    """fp64 output [D] and softmax weights [L_s] of one (sequence, query head)."""
    pr = problem or _Problem(q, k_cache, v_cache, block_tables, seq_lens, scale,
                             num_kv_heads, dtype)
    L = int(pr.sl[s])
    out = np.zeros(pr.D, dtype=np.float64)
    w = np.zeros(max(L, 1), dtype=np.float64)
    if pr.fp8:
        rc = _active().pa_ref_decode_one_fp8(_p(out), _p(w), int(s), int(h), *pr.common(),
                                             *pr.scales())
    else:
        rc = _active().pa_ref_decode_one(_p(out), _p(w), int(s), int(h), *pr.common())
    if rc:
        raise ValueError("oracle decode_one: invalid input")
    return out, w[:L]


def decode_multi(q, k_cache, v_cache, block_tables, seq_lens, query_start, scale,
                 num_kv_heads, dtype: str) -> np.ndarray:
    """fp64 multi-token-query attention: q [T, H_q, D] packed by query_start
    [B+1]; returns [T, H_q, D]."""
    qh = _host(q)
    kc, vc = _host(k_cache), _host(v_cache)
    bt = _host(block_tables, np.int32)
    sl = _host(seq_lens, np.int32)
    qs = _host(query_start, np.int32)
    T, H, D = qh.shape
    N, kvh, bs, _ = kc.shape
    if kvh != num_kv_heads:
        raise ValueError("num_kv_heads does not match the cache")
    out = np.zeros((T, H, D), dtype=np.float64)
    rc = _active().pa_ref_decode_multi(_p(out), _p(qh), _p(kc), _p(vc), _p(bt), _p(sl),
                                       _p(qs), sl.shape[0], H, kvh, D, bs, N, bt.shape[1],
                                       H * D, float(scale), REF_DTYPE[dtype])
    if rc:
        raise ValueError("oracle decode_multi: invalid input")
    return out


def problem(q, k_cache, v_cache, block_tables, seq_lens, scale, num_kv_heads,
            dtype: str, kv_scales=None) -> _Problem:
    """Marshal once, then pass as ``problem=`` to ``decode_one`` /
    ``partition_stats`` for many samples of one large batch."""
    return _Problem(q, k_cache, v_cache, block_tables, seq_lens, scale,
                    num_kv_heads, dtype, kv_scales)


def partition_stats(s, h, partition_size, q, k_cache, v_cache, block_tables,
                    seq_lens, scale, num_kv_heads, dtype: str,
                    problem: _Problem | None = None):
    """(m[P], l[P], o[P, D]) of the split-KV partitions of one (seq, head)."""
    pr = problem or _Problem(q, k_cache, v_cache, block_tables, seq_lens, scale,
                             num_kv_heads, dtype)
    L = int(pr.sl[s])
    P = max(1, -(-L // partition_size))
    m = np.zeros(P); l = np.zeros(P); o = np.zeros((P, pr.D))
    n = _active().pa_ref_partition_stats(_p(m), _p(l), _p(o), int(s), int(h),
                                       int(partition_size), *pr.common())
    if n < 0:
        raise ValueError("oracle partition_stats: invalid input")
    return m[:n], l[:n], o[:n]


def lse_merge(m, l, o) -> np.ndarray:
    m = np.ascontiguousarray(m, np.float64)
    l = np.ascontiguousarray(l, np.float64)
    o = np.ascontiguousarray(o, np.float64)
    out = np.zeros(o.shape[-1], dtype=np.float64)
    _active().pa_ref_lse_merge(_p(out), _p(m), _p(l), _p(o), int(m.shape[0]),
                             int(o.shape[-1]))
    return out
