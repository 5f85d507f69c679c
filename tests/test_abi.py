"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_151_gb300 import build as pabuild
from paged_kv_cache_151_gb300 import pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


def declared_functions():
    text = "".join(open(os.path.join(ROOT, "include", f)).read()
                   for f in sorted(os.listdir(os.path.join(ROOT, "include"))) if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    pabuild.build()
    return pa.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_decode_partitioned",
              "pa_decode_partitioned_workspace_size", "pa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pa.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pa_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_status_strings_and_version(lib):
    assert pa.pa_abi_version() == 4
    assert pa.pa_status_string(0) == "ok"
    assert "invalid" in pa.pa_status_string(-1)
    assert "unsupported" in pa.pa_status_string(-2)
    assert "workspace" in pa.pa_status_string(-3)


def test_workspace_size_formula(lib):
    def up(x):
        return (x + 255) // 256 * 256
    B, H, D, L, P = 8, 64, 128, 131072, 512
    parts = L // P
    rows = B * H * parts
    expect = up(rows * D * 4) + 2 * up(rows * 4)
    assert pa.pa_decode_partitioned_workspace_size(B, H, D, L, P) == expect
    assert pa.pa_decode_partitioned_workspace_size(B, H, D, L, 100) == 0   # not a multiple of 16
    assert pa.pa_decode_partitioned_workspace_size(0, H, D, L, P) == 0


def _decode_status(lib, **kw):
    args = dict(out=1, q=1, k_cache=16, v_cache=16, block_tables=1, seq_lens=1,
                num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=64, num_blocks=10,
                block_size=16, max_blocks=4, q_seq_stride=512, scale=0.125, dtype=0)
    args.update(kw)
    a = args
    return lib.pa_decode(a["out"], a["q"], a["k_cache"], a["v_cache"], a["block_tables"],
                         a["seq_lens"], a["num_seqs"], a["num_heads"], a["num_kv_heads"],
                         a["head_dim"], a["num_blocks"], a["block_size"], a["max_blocks"],
                         a["q_seq_stride"], a["scale"], a["dtype"], None)


def test_host_side_argument_checks(lib):
    # each of these fails its host check before anything is launched
    assert _decode_status(lib, out=None) == -1
    assert _decode_status(lib, num_heads=7) == -1              # not a multiple of H_kv
    assert _decode_status(lib, head_dim=96) == -2
    assert _decode_status(lib, block_size=32) == -2
    assert _decode_status(lib, num_heads=32, num_kv_heads=2, q_seq_stride=32 * 64) == -2  # G=16
    assert _decode_status(lib, dtype=7) == -2
    assert _decode_status(lib, q_seq_stride=100) == -1
    assert _decode_status(lib, k_cache=8) == -1                # not 16-byte aligned
    assert _decode_status(lib, scale=float("nan")) == -1
    assert _decode_status(lib, num_seqs=0) == 0                # nothing to do
    assert _decode_status(lib, num_seqs=-1) == -1
    rc = lib.pa_reshape_and_cache(1, 1, 1, 1, 1, 0, 2, 64, 128, 128, 10, 16, 0, None)
    assert rc == 0                                              # zero tokens
    rc = lib.pa_reshape_and_cache(1, 1, 1, 1, 1, 3, 2, 64, 100, 128, 10, 16, 0, None)
    assert rc == -1                                             # stride < row
    rc = lib.pa_reshape_and_cache(1, 1, 1, 1, 1, 3, 2, 4, 8, 8, 10, 16, 1, None)
    assert rc == -2                                             # 8-byte rows
    ws = ctypes.c_void_p(256)
    rc = lib.pa_decode_partitioned(1, 1, 16, 16, 1, 1, 4, 8, 2, 64, 10, 16, 4, 512,
                                   0.125, 0, 512, 64, ws, 16, None)
    assert rc == -3                                             # workspace too small
    rc = lib.pa_decode_partitioned(1, 1, 16, 16, 1, 1, 4, 8, 2, 64, 10, 16, 4, 512,
                                   0.125, 0, 100, 64, ws, 1 << 20, None)
    assert rc == -1                                             # partition not x16


def _multi_status(lib, **kw):
    a = dict(out=16, q=16, k_cache=16, v_cache=16, block_tables=16, seq_lens=16,
             query_start=16, num_seqs=4, num_q_rows=12, max_query_len=3, num_heads=8,
             num_kv_heads=2, head_dim=64, num_blocks=10, block_size=16, max_blocks=4,
             q_row_stride=512, scale=0.125, dtype=1)
    a.update(kw)
    return lib.pa_decode_multi(a["out"], a["q"], a["k_cache"], a["v_cache"],
                               a["block_tables"], a["seq_lens"], a["query_start"],
                               a["num_seqs"], a["num_q_rows"], a["max_query_len"],
                               a["num_heads"], a["num_kv_heads"], a["head_dim"],
                               a["num_blocks"], a["block_size"], a["max_blocks"],
                               a["q_row_stride"], a["scale"], a["dtype"], None)


def test_multi_query_host_checks(lib):
    assert _multi_status(lib, dtype=0) == -2                   # fp32: not built
    assert _multi_status(lib, query_start=None) == -1
    assert _multi_status(lib, num_q_rows=-1) == -1
    assert _multi_status(lib, max_query_len=-1) == -1
    assert _multi_status(lib, q=8) == -1                       # q not 16-byte aligned
    assert _multi_status(lib, q_row_stride=516) == -1          # rows not 16-byte aligned
    assert _multi_status(lib, head_dim=96) == -2
    assert _multi_status(lib, num_seqs=0) == 0                 # nothing to do
    assert _multi_status(lib, num_q_rows=0) == 0
    assert _multi_status(lib, max_query_len=0) == 0            # no rows can exist


def test_fp8_host_checks(lib):
    P = 16
    # cache write: bad head_dim, unaligned source, null scale, zero tokens
    args = [P, P, P, P, P, P, P, 4, 2, 64, 128, 128, 10, 16, 1, None]
    a = list(args); a[9] = 40
    assert lib.pa_reshape_and_cache_fp8(*a) == -2              # head_dim not x16
    a = list(args); a[0] = 8
    assert lib.pa_reshape_and_cache_fp8(*a) == -1              # k not 16-byte aligned
    a = list(args); a[4] = None
    assert lib.pa_reshape_and_cache_fp8(*a) == -1              # no k_scale
    a = list(args); a[7] = 0
    assert lib.pa_reshape_and_cache_fp8(*a) == 0               # nothing to do
    a = list(args); a[14] = 7
    assert lib.pa_reshape_and_cache_fp8(*a) == -2              # source dtype
    # decode: fp32 q unsupported, null scales, zero sequences
    dec = [P, P, P, P, P, P, P, P, 4, 8, 2, 64, 10, 16, 4, 512, 0.125, 1, None]
    a = list(dec); a[17] = 0
    assert lib.pa_decode_fp8(*a) == -2                         # q in fp32
    a = list(dec); a[4] = None
    assert lib.pa_decode_fp8(*a) == -1
    a = list(dec); a[8] = 0
    assert lib.pa_decode_fp8(*a) == 0
    part = dec[:-1] + [100, 64, ctypes.c_void_p(256), 1 << 20, None]
    assert lib.pa_decode_partitioned_fp8(*part) == -1          # partition not x16
    part = dec[:-1] + [512, 64, ctypes.c_void_p(256), 16, None]
    assert lib.pa_decode_partitioned_fp8(*part) == -3          # workspace too small
    # the 16-bit entry points do not take E4M3 as a dtype
    assert _decode_status(lib, dtype=3) == -2


def test_copy_blocks_host_checks(lib):
    arr = (ctypes.c_void_p * 3)(16, 32, 48)
    assert lib.pa_copy_blocks(arr, 3, 16, 0, 10, 4096, None) == 0        # no pairs
    assert lib.pa_copy_blocks(arr, 0, 16, 5, 10, 4096, None) == 0        # no caches
    assert lib.pa_copy_blocks(arr, 3, 16, 5, 10, 4100, None) == -2       # not x16
    assert lib.pa_copy_blocks(arr, 3, 16, 5, 10, 0, None) == -1
    assert lib.pa_copy_blocks(arr, 3, 16, -1, 10, 4096, None) == -1
    assert lib.pa_copy_blocks(arr, 300, 16, 5, 10, 4096, None) == -2     # too many caches
    assert lib.pa_copy_blocks(arr, 3, None, 5, 10, 4096, None) == -1     # no mapping
    bad = (ctypes.c_void_p * 2)(16, 24)                                  # unaligned cache
    assert lib.pa_copy_blocks(bad, 2, 16, 5, 10, 4096, None) == -1


def _partitioned_status(lib, noalloc, **kw):
    """Status of pa_decode_partitioned (with a workspace of `ws_bytes`) or of
    pa_decode_partitioned_noalloc for the same arguments."""
    a = dict(out=16, q=16, k_cache=16, v_cache=16, block_tables=16, seq_lens=16,
             num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=64, num_blocks=10,
             block_size=16, max_blocks=4, q_seq_stride=512, scale=0.125, dtype=1,
             partition_size=512, max_seq_len=64, ws_bytes=1 << 30)
    a.update(kw)
    head = [a["out"], a["q"], a["k_cache"], a["v_cache"], a["block_tables"], a["seq_lens"],
            a["num_seqs"], a["num_heads"], a["num_kv_heads"], a["head_dim"], a["num_blocks"],
            a["block_size"], a["max_blocks"], a["q_seq_stride"], a["scale"], a["dtype"],
            a["partition_size"], a["max_seq_len"]]
    if noalloc:
        return lib.pa_decode_partitioned_noalloc(*head, None)
    return lib.pa_decode_partitioned(*head, ctypes.c_void_p(256), a["ws_bytes"], None)


@pytest.mark.parametrize("bad", [
    dict(num_seqs=0, partition_size=7),            # nothing to do, but a bad partition
    dict(num_seqs=0, num_heads=0),                 # nothing to do, but no heads
    dict(num_seqs=0, max_seq_len=-1),
    dict(out=None),
    dict(head_dim=96),
    dict(partition_size=100),
    dict(num_heads=7),
    dict(out=None, max_seq_len=1 << 24),           # null pointers on a huge problem
    dict(num_seqs=0),                              # valid and empty: PA_OK from both
])
def test_noalloc_refuses_bad_arguments_like_the_workspace_call(lib, bad):
    """Both split-KV entry points check their arguments in the same order, so
    a bad input gets the same status from each; none of these reaches a GPU."""
    assert (_partitioned_status(lib, True, **bad) ==
            _partitioned_status(lib, False, **bad))


def test_workspace_size_overflow_is_refused(lib):
    """num_seqs * num_heads * partitions * head_dim * 4 past 2^64 gives 0
    (invalid), not a wrapped size that a workspace check could accept."""
    assert pa.pa_decode_partitioned_workspace_size(65535, 8 * 65535, 128, 2**31 - 1, 16) == 0
    rows = 65535 * 8 * (2**27)                     # large, but no product overflows
    up = lambda x: (x + 255) // 256 * 256
    assert (pa.pa_decode_partitioned_workspace_size(65535, 8, 128, 2**31 - 1, 16) ==
            up(rows * 128 * 4) + 2 * up(rows * 4))


def test_noalloc_limit_matches_the_header():
    text = open(HEADER).read()
    m = re.search(r"#define\s+PA_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "PA_NOALLOC_SCRATCH_BYTES not found in include/pa.h"
    assert pa.PA_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def _cascade_status(lib, **kw):
    a = dict(out=16, q=16, k_cache=16, v_cache=16, prefix=16, n_prefix=8, block_tables=16,
             seq_lens=16, num_seqs=4, num_heads=8, num_kv_heads=2, head_dim=64, num_blocks=100,
             block_size=16, max_blocks=4, q_seq_stride=512, scale=0.125, dtype=1,
             ws=256, ws_bytes=1 << 30)
    a.update(kw)
    return lib.pa_decode_cascade(a["out"], a["q"], a["k_cache"], a["v_cache"], a["prefix"],
                                 a["n_prefix"], a["block_tables"], a["seq_lens"], a["num_seqs"],
                                 a["num_heads"], a["num_kv_heads"], a["head_dim"],
                                 a["num_blocks"], a["block_size"], a["max_blocks"],
                                 a["q_seq_stride"], a["scale"], a["dtype"],
                                 ctypes.c_void_p(a["ws"]), a["ws_bytes"], None)


def test_cascade_host_checks(lib):
    """Refusals of pa_decode_cascade that come before any launch."""
    assert _cascade_status(lib, prefix=None) == -1            # no prefix list
    assert _cascade_status(lib, n_prefix=-1) == -1
    assert _cascade_status(lib, dtype=0) == -2                # fp32 with a prefix
    assert _cascade_status(lib, ws_bytes=16) == -3            # workspace too small
    assert _cascade_status(lib, ws=None) == -3
    assert _cascade_status(lib, ws=128) == -3                 # not 256-byte aligned
    assert _cascade_status(lib, q=8) == -1                    # q not 16-byte aligned
    assert _cascade_status(lib, num_seqs=0) == 0              # nothing to do
    assert _cascade_status(lib, head_dim=96) == -2


def test_cascade_workspace_size(lib):
    def up(x):
        return (x + 255) // 256 * 256
    # 128 prefix blocks: chunks of 32 blocks -> 4 parts; 32 own blocks -> 1 part of 512 tokens
    B, H, D = 128, 32, 128
    rows = B * H * (4 + 1)
    assert pa.pa_decode_cascade_workspace_size(B, H, D, 128, 32) == \
        up(rows * D * 4) + 2 * up(rows * 4)
    # 300 prefix blocks: chunks of 32 -> 10 parts; 70 own blocks -> 3 parts of 512 tokens
    rows = 2 * 8 * (10 + 3)
    assert pa.pa_decode_cascade_workspace_size(2, 8, 64, 300, 70) == \
        up(rows * 64 * 4) + 2 * up(rows * 4)
    # 1000 prefix blocks: chunks of 64 (at most 16 chunks)
    rows = 2 * 8 * (16 + 1)
    assert pa.pa_decode_cascade_workspace_size(2, 8, 64, 1000, 1) == \
        up(rows * 64 * 4) + 2 * up(rows * 4)
    assert pa.pa_decode_cascade_workspace_size(B, H, D, 0, 32) == 0


def test_cascade_refuses_more_prefix_items_than_an_int_counts(lib):
    # 16 chunks x 65535 KV heads x 4096 row groups of 128 rows: past 2^31 items
    assert _cascade_status(lib, num_seqs=65535, num_heads=8 * 65535, num_kv_heads=65535,
                           n_prefix=10000, q_seq_stride=8 * 65535 * 64) == -2
