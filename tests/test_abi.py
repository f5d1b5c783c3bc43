"""The C ABI without a GPU: libfa.so builds, loads, exports every function that
include/fa.h declares, and rejects bad arguments on the host before any CUDA
call (so these run on a CPU-only machine)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_05_gb300 import build
    so = build.build()
    return ctypes.CDLL(so)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_fwd_f32", "fa_bwd_workspace_bytes", "fa_sync_status", "fa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def _fwd(lib):
    f = lib.fa_fwd
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, fl, vp]
    f.restype = i
    return f


def test_status_strings(lib):
    lib.fa_status_string.restype = ctypes.c_char_p
    seen = set()
    for s in range(5):
        txt = lib.fa_status_string(s).decode()
        assert txt and txt not in seen
        seen.add(txt)
    assert lib.fa_status_string(99).decode() == "unknown status"


def test_host_validation_without_gpu(lib):
    f = _fwd(lib)
    p = 1 << 20   # a fake, 16-byte aligned address: never dereferenced on these paths
    assert f(p, p + 4096, p + 8192, p + 12288, p + 16384, 1, 1, 8, 8, 64, 0, float("nan"), None) == 1
    assert f(p, p + 4096, p + 8192, p + 12288, p + 16384, 1, 1, 8, 8, 64, 0, -0.5, None) == 1
    assert f(p, p + 4096, p + 8192, p + 12288, p + 16384, 1, 1, 8, 8, 64, 2, 0.5, None) == 1
    assert f(p, p + 4096, p + 8192, p + 12288, p + 16384, 1, 1, 8, 8, 96, 0, 0.5, None) == 2
    assert f(p, p + 4096, p + 8192, p + 12288, p + 16384, -1, 1, 8, 8, 64, 0, 0.5, None) == 1
    assert f(p, p, p + 8192, p + 12288, p + 16384, 1, 1, 8, 8, 64, 0, 0.5, None) in (1, 2, 3)
    # empty problems are a no-op that touches nothing
    assert f(None, None, None, None, None, 0, 4, 8, 8, 64, 0, 0.5, None) == 0
    assert f(None, None, None, None, None, 1, 1, 0, 8, 128, 1, 0.5, None) == 0
    # null or misaligned pointers
    assert f(None, p, p, p, p, 1, 1, 8, 8, 64, 0, 0.5, None) == 1
    assert f(p + 2, p + 4096, p + 8192, p + 12288, p + 16384, 1, 1, 8, 8, 64, 0, 0.5, None) == 1
    # output overlapping an input
    assert f(p, p + 4096, p + 8192, p + 100, p + 16384, 1, 1, 8, 8, 64, 0, 0.5, None) == 1


def test_bwd_workspace_and_validation(lib):
    lib.fa_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    ws = lib.fa_bwd_workspace_bytes(8, 32, 4096, 4096, 128)
    rows = 8 * 32 * 4096
    # + the fixed-point bounds of the deterministic mode: 2 floats per head, 1 int per query block
    assert ws == 2 * rows * 4 + rows * 128 * 4 + (8 * 32 * 2 * 4 + rows // 128 * 4)
    assert lib.fa_bwd_workspace_bytes(1, 1, 1, 1, 64) == 2 * 512 + 128 * 64 * 4 + 256   # rows padded to 128
    assert lib.fa_bwd_workspace_bytes(1, 1, 8, 8, 96) == 0
    b = lib.fa_bwd
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    b.argtypes = [vp] * 9 + [i] * 6 + [fl, vp, ctypes.c_size_t, vp]
    b.restype = i
    p = 1 << 20
    ptrs = [p + 4096 * n for n in range(9)]
    assert b(*ptrs, 1, 1, 8, 8, 256, 0, 0.5, p + 65536, 1 << 20, None) == 2    # d=256 backward
    assert b(*ptrs, 1, 1, 8, 8, 64, 0, 0.5, p + 65536, 16, None) == 1          # workspace too small
    assert b(*ptrs, 1, 1, 8, 8, 64, 0, 0.5, None, 1 << 20, None) == 1          # no workspace
    assert b(*ptrs, 0, 1, 8, 8, 64, 0, 0.5, None, 0, None) == 0                 # empty


def test_decode_workspace_and_validation(lib):
    lib.fa_decode_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.fa_decode_workspace_bytes.restype = ctypes.c_size_t
    # 1024 tiles of 32 keys, 256 heads: 8 chunks per head (2048 chunks in all), 130 floats per row state
    assert lib.fa_decode_workspace_bytes(8, 32, 1, 32768, 128) == 256 * 8 * 1 * 130 * 4
    # at least 8 tiles a chunk: 4 tiles -> one chunk; 2 rows x 66 floats, rounded up to 256 bytes
    assert lib.fa_decode_workspace_bytes(1, 1, 2, 100, 64) == 768
    assert lib.fa_decode_workspace_bytes(1, 1, 17, 64, 128) == 0     # too many query rows
    assert lib.fa_decode_workspace_bytes(1, 1, 9, 64, 256) == 0
    assert lib.fa_decode_workspace_bytes(1, 1, 8, 64, 96) == 0       # head width
    f = lib.fa_decode
    vp, i, fl, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, fl, vp, sz, vp]
    f.restype = i
    p = 1 << 20   # fake aligned addresses, never dereferenced on these paths
    args = (p, p + (1 << 16), p + (2 << 16), p + (3 << 16), p + (4 << 16))
    assert f(*args, 1, 1, 4, 64, 128, 1, float("inf"), p + (5 << 16), 1 << 16, None) == 1
    assert f(*args, 1, 1, 4, 64, 128, 2, 0.1, p + (5 << 16), 1 << 16, None) == 1      # causal flag
    assert f(*args, 1, 1, 17, 64, 128, 1, 0.1, p + (5 << 16), 1 << 16, None) in (2, 3)   # no sm_103 here: 3


def test_fp8_host_validation(lib):
    """FP8 entry points reject bad sizes before any device work (no GPU needed)."""
    import ctypes
    vp = ctypes.c_void_p
    lib.fa_fp8_vt_stride.argtypes = [ctypes.c_int]
    lib.fa_fp8_vt_stride.restype = ctypes.c_size_t
    assert [lib.fa_fp8_vt_stride(t) for t in (0, 1, 16, 17, 4096)] == [0, 16, 16, 32, 4096]
    lib.fa_fwd_fp8.argtypes = [vp] * 8 + [ctypes.c_int] * 6 + [ctypes.c_float, vp]
    lib.fa_fwd_fp8.restype = ctypes.c_int
    lib.fa_fp8_quantize.argtypes = [vp] * 4 + [ctypes.c_int] * 5 + [vp] * 6 + [vp]
    lib.fa_fp8_quantize.restype = ctypes.c_int
    p = ctypes.c_void_p(1 << 20)        # aligned, never dereferenced: every call fails validation first
    args8 = [p] * 8
    assert lib.fa_fwd_fp8(*args8, 1, 1, 64, 64, 64, 0, 0.1, None) == 2          # d = 64: unsupported
    assert lib.fa_fwd_fp8(*args8, 1, 1, 64, 64, 96, 0, 0.1, None) == 2          # d = 96
    assert lib.fa_fwd_fp8(*args8, 1, 1, 64, 64, 128, 2, 0.1, None) == 1         # causal flag
    assert lib.fa_fwd_fp8(*args8, 1, 1, 64, 64, 128, 0, -1.0, None) == 1        # scale
    assert lib.fa_fwd_fp8(None, *args8[1:], 1, 1, 64, 64, 128, 0, 0.1, None) == 1
    assert lib.fa_fwd_fp8(*args8[:7], ctypes.c_void_p((1 << 20) + 4), 1, 1, 64, 64, 128, 0, 0.1, None) == 1
    assert lib.fa_fwd_fp8(*args8, 1, 1, 0, 64, 128, 0, 0.1, None) == 0          # nothing to do
    q = [p] * 3
    outs = [ctypes.c_void_p((1 << 21) + (i << 24)) for i in range(6)]
    assert lib.fa_fp8_quantize(*q, None, 1, 1, 64, 64, 100, *outs, None) == 2    # d
    assert lib.fa_fp8_quantize(*q, None, -1, 1, 64, 64, 128, *outs, None) == 1
    assert lib.fa_fp8_quantize(*q, ctypes.c_void_p((1 << 20) + 8), 1, 1, 64, 64, 128, *outs, None) == 1
    overlap = [outs[0], outs[0]] + outs[2:]
    assert lib.fa_fp8_quantize(*q, None, 1, 1, 64, 64, 128, *overlap, None) == 1
    assert lib.fa_fp8_quantize(*q, None, 1, 1, 0, 0, 128, *outs, None) == 0


def _noalloc(lib):
    f = lib.fa_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 9 + [i] * 6 + [ctypes.c_float, vp]
    f.restype = i
    return f


def _far_apart(n, base=1 << 40, step=1 << 34):
    """Fake, aligned, non-overlapping device addresses, never dereferenced on these paths."""
    return [base + step * i for i in range(n)]


def test_noalloc_scratch_examples_in_header(lib):
    """The sizes include/fa.h names as fitting the 64 MiB scratch do fit; the one it names
    as not fitting does not."""
    lib.fa_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    text = open(HEADER).read()
    limit = int(re.search(r"#define FA_BWD_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text).expand(r"\1")) << 20
    assert limit == 64 << 20
    for B, H, T, d in ((8, 8, 1920, 128), (1, 32, 3840, 128), (8, 16, 1920, 64)):
        assert f"B{B} H{H} T{T}" in text
        assert lib.fa_bwd_workspace_bytes(B, H, T, T, d) <= limit, (B, H, T, d)
    assert "not B8 H8 T2048" in text
    assert lib.fa_bwd_workspace_bytes(8, 8, 2048, 2048, 128) > limit
    # the row figures the header quotes: per-row bytes and the largest row counts
    per_row = {128: 520, 64: 264}
    for d, rows in ((128, 129_000), (64, 254_000)):
        assert abs(limit / per_row[d] - rows) < 0.01 * rows


def test_noalloc_checks_arguments_before_its_scratch_limit(lib):
    """fa_bwd_noalloc reports fa_bwd's argument errors even for sizes beyond its scratch,
    and only then FA_ERR_UNSUPPORTED for the size; none of this makes a CUDA call."""
    f = _noalloc(lib)
    ptrs = _far_apart(9)
    big = (8, 32, 4096, 4096, 128)
    assert f(*ptrs, *big, 1, 0.088, None) == 2                      # beyond the scratch
    assert f(*ptrs, *big, 1, float("nan"), None) == 1               # bad scale
    assert f(*ptrs, *big, 2, 0.088, None) == 1                      # bad causal flag
    assert f(None, *ptrs[1:], *big, 1, 0.088, None) == 1            # null q
    assert f(ptrs[0] + 2, *ptrs[1:], *big, 1, 0.088, None) == 1     # misaligned q
    assert f(*ptrs[:6], ptrs[0], *ptrs[7:], *big, 1, 0.088, None) == 1   # dq overlaps q
    assert f(*ptrs, 8, 32, 4096, 4096, 256, 1, 0.088, None) == 2    # d = 256 backward


def test_bwd_workspace_bytes_rejects_head_overflow(lib):
    lib.fa_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 5
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    assert lib.fa_bwd_workspace_bytes(1 << 16, 1 << 16, 1, 1, 64) == 0   # B*H beyond 32 bits
    assert lib.fa_bwd_workspace_bytes(1 << 15, 1 << 15, 1, 1, 64) > 0
