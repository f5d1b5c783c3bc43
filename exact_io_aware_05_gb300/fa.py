"""ctypes binding of libfa.so (include/fa.h): argument marshalling only.

Every function here checks tensor dtypes, shapes, devices and contiguity,
reads the current CUDA stream, and calls the C entry point of the same name
with raw device pointers.  No attention arithmetic happens in Python and
there is no fallback: importing this module fails if libfa.so is missing,
and every nonzero status raises ``FAError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run exact_io_aware_05_gb300.build.build() "
                      "(or __graft_entry__.build()) first")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_lib.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]
_lib.fa_fwd.restype = _i
_lib.fa_fwd_f32.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]
_lib.fa_fwd_f32.restype = _i
_lib.fa_fwd_masked.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _i, _f, _vp]
_lib.fa_fwd_masked.restype = _i
_lib.fa_bwd_masked.argtypes = [_vp] * 9 + [_i] * 7 + [_vp, _i, _i, _f, _vp, _sz, _vp]
_lib.fa_bwd_masked.restype = _i
_lib.fa_fp8_vt_stride.argtypes = [_i]
_lib.fa_fp8_vt_stride.restype = _sz
_lib.fa_fp8_quantize.argtypes = [_vp] * 4 + [_i] * 5 + [_vp] * 6 + [_vp]
_lib.fa_fp8_quantize.restype = _i
_lib.fa_fwd_fp8.argtypes = [_vp] * 8 + [_i] * 6 + [_f, _vp]
_lib.fa_fwd_fp8.restype = _i
_lib.fa_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]
_lib.fa_decode.restype = _i
_lib.fa_decode_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
_lib.fa_decode_workspace_bytes.restype = _sz
_lib.fa_bwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
_lib.fa_bwd_workspace_bytes.restype = _sz
_lib.fa_bwd.argtypes = [_vp] * 9 + [_i] * 6 + [_f, _vp, _sz, _vp]
_lib.fa_bwd.restype = _i
_lib.fa_bwd_deterministic.argtypes = [_vp] * 9 + [_i] * 6 + [_f, _vp, _sz, _vp]
_lib.fa_bwd_deterministic.restype = _i
_lib.fa_bwd_stage.argtypes = [_i] + [_vp] * 9 + [_i] * 6 + [_f, _vp, _sz, _vp]
_lib.fa_bwd_stage.restype = _i
_lib.fa_bwd_noalloc.argtypes = [_vp] * 9 + [_i] * 6 + [_f, _vp]
_lib.fa_bwd_noalloc.restype = _i
_lib.fa_sync_status.argtypes = [_vp]
_lib.fa_sync_status.restype = _i
_lib.fa_status_string.argtypes = [_i]
_lib.fa_status_string.restype = ctypes.c_char_p

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)


class FAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {_lib.fa_status_string(status).decode()} (status {status})")


def lib() -> ctypes.CDLL:
    return _lib


def _check(fn: str, st: int) -> None:
    if st != FA_OK:
        raise FAError(fn, st)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple, device: torch.device) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _shapes(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k must be [B, H, T, d]")
    B, H, Tq, d = q.shape
    Tk = k.shape[2]
    return B, H, Tq, Tk, d


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """O and lse for bf16 q [B,H,Tq,d], k/v [B,H,Tk,d]; o bf16 like q, lse f32 [B,H,Tq]."""
    B, H, Tq, Tk, d = _shapes(q, k)
    dev = q.device
    _need(q, "q", torch.bfloat16, (B, H, Tq, d), dev)
    _need(k, "k", torch.bfloat16, (B, H, Tk, d), dev)
    _need(v, "v", torch.bfloat16, (B, H, Tk, d), dev)
    _need(o, "o", torch.bfloat16, (B, H, Tq, d), dev)
    _need(lse, "lse", torch.float32, (B, H, Tq), dev)
    _check("fa_fwd", _lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Tq, Tk, d,
                                 int(bool(causal)), float(scale), _stream(stream)))


def _block_mask(block_mask, B, H, Tq, Tk, dev):
    """(pointer, per_head) of a block mask: a uint8/bool tensor on `dev` shaped
    [ceil(Tq/128), ceil(Tk/128)] (all heads) or [B, H, ceil(Tq/128), ceil(Tk/128)]."""
    if block_mask is None:
        return None, 0
    nq, nk = -(-Tq // 128), -(-Tk // 128)
    if block_mask.device != dev or block_mask.dtype not in (torch.uint8, torch.bool) or \
            not block_mask.is_contiguous():
        raise ValueError("block_mask: contiguous uint8 or bool tensor on the inputs' device")
    if tuple(block_mask.shape) == (nq, nk):
        return block_mask.data_ptr(), 0
    if tuple(block_mask.shape) == (B, H, nq, nk):
        return block_mask.data_ptr(), 1
    raise ValueError(f"block_mask: shape ({nq}, {nk}) or ({B}, {H}, {nq}, {nk}), got {tuple(block_mask.shape)}")


def fa_fwd_masked(q, k, v, o, lse, window=(-1, -1), block_mask=None, scale: float = 1.0, stream=None) -> None:
    """fa_fwd under a window (left, right) around the bottom-right diagonal (-1 = unbounded
    side; (-1, 0) is causal) and an optional 128 x 128 block mask."""
    B, H, Tq, Tk, d = _shapes(q, k)
    dev = q.device
    _need(q, "q", torch.bfloat16, (B, H, Tq, d), dev)
    _need(k, "k", torch.bfloat16, (B, H, Tk, d), dev)
    _need(v, "v", torch.bfloat16, (B, H, Tk, d), dev)
    _need(o, "o", torch.bfloat16, (B, H, Tq, d), dev)
    _need(lse, "lse", torch.float32, (B, H, Tq), dev)
    bm, per_head = _block_mask(block_mask, B, H, Tq, Tk, dev)
    _check("fa_fwd_masked", _lib.fa_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Tq, Tk, d,
                                               int(window[0]), int(window[1]), bm, per_head, float(scale),
                                               _stream(stream)))


def fa_decode_workspace_bytes(B: int, H: int, Tq: int, Tk: int, d: int) -> int:
    return int(_lib.fa_decode_workspace_bytes(B, H, Tq, Tk, d))


def fa_decode(q, k, v, o, lse, causal: bool, scale: float, workspace: torch.Tensor, stream=None) -> None:
    """Split-KV O and lse (as fa_fwd) for Tq <= 16 (d = 64, 128) or 8 (d = 256) query rows."""
    B, H, Tq, Tk, d = _shapes(q, k)
    dev = q.device
    _need(q, "q", torch.bfloat16, (B, H, Tq, d), dev)
    _need(k, "k", torch.bfloat16, (B, H, Tk, d), dev)
    _need(v, "v", torch.bfloat16, (B, H, Tk, d), dev)
    _need(o, "o", torch.bfloat16, (B, H, Tq, d), dev)
    _need(lse, "lse", torch.float32, (B, H, Tq), dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace: must be a contiguous tensor on the same device")
    nbytes = workspace.numel() * workspace.element_size()
    _check("fa_decode", _lib.fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Tq, Tk, d,
                                       int(bool(causal)), float(scale), _ptr(workspace), nbytes,
                                       _stream(stream)))


def attention_decode(q, k, v, causal: bool, scale: float, workspace=None, stream=None):
    """Allocates O, lse (and the workspace if not given) and runs fa_decode."""
    B, H, Tq, Tk, d = _shapes(q, k)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = fa_decode_workspace_bytes(B, H, Tq, Tk, d)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    fa_decode(q, k, v, o, lse, causal, scale, workspace, stream)
    return o, lse


def fa_fwd_f32(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """fp32 SIMT forward (precision reference path); all tensors float32."""
    B, H, Tq, Tk, d = _shapes(q, k)
    dev = q.device
    _need(q, "q", torch.float32, (B, H, Tq, d), dev)
    _need(k, "k", torch.float32, (B, H, Tk, d), dev)
    _need(v, "v", torch.float32, (B, H, Tk, d), dev)
    _need(o, "o", torch.float32, (B, H, Tq, d), dev)
    _need(lse, "lse", torch.float32, (B, H, Tq), dev)
    _check("fa_fwd_f32", _lib.fa_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Tq, Tk,
                                         d, int(bool(causal)), float(scale), _stream(stream)))


def fa_bwd_workspace_bytes(B: int, H: int, Tq: int, Tk: int, d: int) -> int:
    return int(_lib.fa_bwd_workspace_bytes(B, H, Tq, Tk, d))


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, causal: bool, scale: float, workspace: torch.Tensor,
           stream=None) -> None:
    """dQ, dK, dV (bf16) from bf16 q, k, v, o, dO and the f32 lse of fa_fwd."""
    _bwd_call("fa_bwd", q, k, v, o, lse, dO, dq, dk, dv, causal, scale, workspace, stream)


def fa_bwd_deterministic(q, k, v, o, lse, dO, dq, dk, dv, causal: bool, scale: float,
                         workspace: torch.Tensor, stream=None) -> None:
    """fa_bwd with the dQ additions in a fixed order: dq is bitwise reproducible."""
    _bwd_call("fa_bwd_deterministic", q, k, v, o, lse, dO, dq, dk, dv, causal, scale, workspace, stream)


def _bwd_call(entry, q, k, v, o, lse, dO, dq, dk, dv, causal, scale, workspace, stream):
    B, H, Tq, Tk, d = _shapes(q, k)
    dev = q.device
    for name, t, shp in (("q", q, (B, H, Tq, d)), ("k", k, (B, H, Tk, d)), ("v", v, (B, H, Tk, d)),
                         ("o", o, (B, H, Tq, d)), ("dO", dO, (B, H, Tq, d)), ("dq", dq, (B, H, Tq, d)),
                         ("dk", dk, (B, H, Tk, d)), ("dv", dv, (B, H, Tk, d))):
        _need(t, name, torch.bfloat16, shp, dev)
    _need(lse, "lse", torch.float32, (B, H, Tq), dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace: must be a contiguous tensor on the same device")
    nbytes = workspace.numel() * workspace.element_size()
    _check(entry, getattr(_lib, entry)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                       _ptr(dk), _ptr(dv), B, H, Tq, Tk, d, int(bool(causal)), float(scale),
                                       _ptr(workspace), nbytes, _stream(stream)))


def fa_bwd_stage(stage: int, q, k, v, o, lse, dO, dq, dk, dv, causal: bool, scale: float,
                 workspace: torch.Tensor, stream=None) -> None:
    """Stage 1, 2 or 3 of fa_bwd (preprocess, tile loop, dQ finish); same arguments."""
    B, H, Tq, Tk, d = _shapes(q, k)
    nbytes = workspace.numel() * workspace.element_size()
    _check("fa_bwd_stage", _lib.fa_bwd_stage(int(stage), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                             _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), B, H, Tq, Tk, d,
                                             int(bool(causal)), float(scale), _ptr(workspace), nbytes,
                                             _stream(stream)))


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, causal: bool, scale: float, stream=None) -> None:
    """fa_bwd without a workspace argument, for callers that cannot allocate device memory:
    the scratch is a fixed array inside the library (see include/fa.h for its size limit
    and for why overlapping calls on one device must not be issued)."""
    B, H, Tq, Tk, d = _shapes(q, k)
    _check("fa_bwd_noalloc", _lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, Tq, Tk, d,
                                                 int(bool(causal)), float(scale), _stream(stream)))


def fa_sync_status(stream=None) -> int:
    return int(_lib.fa_sync_status(_stream(stream)))


def fa_status_string(status: int) -> str:
    return _lib.fa_status_string(status).decode()


# ---------------------------------------------------------------- conveniences
def attention_forward(q, k, v, causal: bool, scale: float, stream=None, window=None, block_mask=None):
    """Allocates O and lse with torch and runs fa_fwd (bf16) or fa_fwd_f32 (float32); with a
    window (which replaces `causal`) or a block mask, fa_fwd_masked."""
    B, H, Tq, Tk, d = _shapes(q, k)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    if window is not None or block_mask is not None:
        if window is None:
            window = (-1, 0 if causal else -1)
        elif causal:
            raise ValueError("give either causal or a window")
        fa_fwd_masked(q, k, v, o, lse, window, block_mask, scale, stream)
    else:
        (fa_fwd_f32 if q.dtype == torch.float32 else fa_fwd)(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def fa_fp8_vt_stride(Tk: int) -> int:
    return int(_lib.fa_fp8_vt_stride(Tk))


class FP8Operands(dict):
    """Output of fa_fp8_quantize: q8, k8 [B,H,T,d] and vt8 [B,H,d,ld] e4m3 codes (uint8),
    q_descale [B,H,ceil(Tq/128)], k_descale [B,H,ceil(Tk/128)], v_descale [B,H,d] (f32)."""


def alloc_fp8(B, H, Tq, Tk, d, device) -> FP8Operands:
    u8, f32 = torch.uint8, torch.float32
    return FP8Operands(
        q8=torch.empty((B, H, Tq, d), dtype=u8, device=device),
        k8=torch.empty((B, H, Tk, d), dtype=u8, device=device),
        vt8=torch.empty((B, H, d, fa_fp8_vt_stride(Tk)), dtype=u8, device=device),
        q_descale=torch.empty((B, H, -(-Tq // 128)), dtype=f32, device=device),
        k_descale=torch.empty((B, H, -(-Tk // 128)), dtype=f32, device=device),
        v_descale=torch.empty((B, H, d), dtype=f32, device=device))


def _need_fp8(x: FP8Operands, B, H, Tq, Tk, d, dev):
    _need(x["q8"], "q8", torch.uint8, (B, H, Tq, d), dev)
    _need(x["k8"], "k8", torch.uint8, (B, H, Tk, d), dev)
    _need(x["vt8"], "vt8", torch.uint8, (B, H, d, fa_fp8_vt_stride(Tk)), dev)
    _need(x["q_descale"], "q_descale", torch.float32, (B, H, -(-Tq // 128)), dev)
    _need(x["k_descale"], "k_descale", torch.float32, (B, H, -(-Tk // 128)), dev)
    _need(x["v_descale"], "v_descale", torch.float32, (B, H, d), dev)


def fa_fp8_quantize(q, k, v, signs=None, out: FP8Operands = None, stream=None) -> FP8Operands:
    """e4m3 codes and dequantization factors of bf16 q, k, v (rotated by `signs`, a
    float32 [d] tensor of +-1 on the device, when given)."""
    B, H, Tq, Tk, d = _shapes(q, k)
    dev = q.device
    _need(q, "q", torch.bfloat16, (B, H, Tq, d), dev)
    _need(k, "k", torch.bfloat16, (B, H, Tk, d), dev)
    _need(v, "v", torch.bfloat16, (B, H, Tk, d), dev)
    if signs is not None:
        _need(signs, "signs", torch.float32, (d,), dev)
    x = alloc_fp8(B, H, Tq, Tk, d, dev) if out is None else out
    _need_fp8(x, B, H, Tq, Tk, d, dev)
    _check("fa_fp8_quantize", _lib.fa_fp8_quantize(
        _ptr(q), _ptr(k), _ptr(v), _ptr(signs), B, H, Tq, Tk, d, _ptr(x["q8"]), _ptr(x["k8"]), _ptr(x["vt8"]),
        _ptr(x["q_descale"]), _ptr(x["k_descale"]), _ptr(x["v_descale"]), _stream(stream)))
    return x


def fa_fwd_fp8(x: FP8Operands, o, lse, causal: bool, scale: float, stream=None) -> None:
    """O (bf16) and lse (f32) of attention over the dequantized FP8 operands."""
    B, H, Tq, d = x["q8"].shape
    Tk = x["k8"].shape[2]
    dev = x["q8"].device
    _need_fp8(x, B, H, Tq, Tk, d, dev)
    _need(o, "o", torch.bfloat16, (B, H, Tq, d), dev)
    _need(lse, "lse", torch.float32, (B, H, Tq), dev)
    _check("fa_fwd_fp8", _lib.fa_fwd_fp8(
        _ptr(x["q8"]), _ptr(x["k8"]), _ptr(x["vt8"]), _ptr(x["q_descale"]), _ptr(x["k_descale"]),
        _ptr(x["v_descale"]), _ptr(o), _ptr(lse), B, H, Tq, Tk, d, int(bool(causal)), float(scale),
        _stream(stream)))


def attention_forward_fp8(q, k, v, causal: bool, scale: float, signs=None, stream=None):
    """fa_fp8_quantize then fa_fwd_fp8; returns (o, lse, the FP8 operands)."""
    x = fa_fp8_quantize(q, k, v, signs, stream=stream)
    B, H, Tq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    fa_fwd_fp8(x, o, lse, causal, scale, stream)
    return o, lse, x


def alloc_workspace(B, H, Tq, Tk, d, device) -> torch.Tensor:
    n = fa_bwd_workspace_bytes(B, H, Tq, Tk, d)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def fa_bwd_masked(q, k, v, o, lse, dO, dq, dk, dv, window=(-1, -1), block_mask=None, deterministic=False,
                  scale: float = 1.0, workspace: torch.Tensor = None, stream=None) -> None:
    """Backward of fa_fwd_masked under the same window and block mask."""
    B, H, Tq, Tk, d = _shapes(q, k)
    dev = q.device
    for name, t, shp in (("q", q, (B, H, Tq, d)), ("k", k, (B, H, Tk, d)), ("v", v, (B, H, Tk, d)),
                         ("o", o, (B, H, Tq, d)), ("dO", dO, (B, H, Tq, d)), ("dq", dq, (B, H, Tq, d)),
                         ("dk", dk, (B, H, Tk, d)), ("dv", dv, (B, H, Tk, d))):
        _need(t, name, torch.bfloat16, shp, dev)
    _need(lse, "lse", torch.float32, (B, H, Tq), dev)
    if workspace is None or workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace: a contiguous tensor on the same device")
    bm, per_head = _block_mask(block_mask, B, H, Tq, Tk, dev)
    nbytes = workspace.numel() * workspace.element_size()
    _check("fa_bwd_masked", _lib.fa_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                               _ptr(dk), _ptr(dv), B, H, Tq, Tk, d, int(window[0]), int(window[1]),
                                               bm, per_head, int(bool(deterministic)), float(scale),
                                               _ptr(workspace), nbytes, _stream(stream)))


def attention_backward(q, k, v, o, lse, dO, causal: bool, scale: float, workspace=None, stream=None,
                       deterministic: bool = False, window=None, block_mask=None):
    """Allocates dQ, dK, dV (and the workspace if not given) and runs fa_bwd
    (fa_bwd_deterministic when `deterministic`; fa_bwd_masked with a window, which
    replaces `causal`, or a block mask)."""
    B, H, Tq, Tk, d = _shapes(q, k)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = alloc_workspace(B, H, Tq, Tk, d, q.device) if workspace is None else workspace
    if window is not None or block_mask is not None:
        if window is None:
            window = (-1, 0 if causal else -1)
        elif causal:
            raise ValueError("give either causal or a window")
        fa_bwd_masked(q, k, v, o, lse, dO, dq, dk, dv, window, block_mask, deterministic, scale, ws, stream)
    else:
        (fa_bwd_deterministic if deterministic else fa_bwd)(q, k, v, o, lse, dO, dq, dk, dv, causal, scale, ws,
                                                            stream)
    return dq, dk, dv
