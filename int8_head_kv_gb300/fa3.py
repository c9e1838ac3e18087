"""Thin Python binding of libfa3.so (the C ABI declared in include/fa3.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the
library has not been built, every call raises; there is no fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from collections import OrderedDict
from typing import Optional

import torch

from . import build as _build

_lib = None

FA3_DEVERR_POS = 1
FA3_DEVERR_LENS = 2
FA3_DEVERR_TIMEOUT = 4
FA3_DEVERR_PAGE = 8
FA3_DEVERR_CALIB = 16


class FA3Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {lib().fa3_status_string(status).decode()} (status {status})")
        self.status = status


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_D = ctypes.c_double

_SIGS = {
    "fa3_status_string": (ctypes.c_char_p, [_I]),
    "fa3_version": (_I, []),
    "fa3_set_kernel_timing": (_I, [_P, _P]),
    "fa3_calibrate_workspace_size": (_SZ, [_I]),
    "fa3_calibrate_perhead": (_I, [_P, _I64, _I, _I64, _I64, _I64, _D, _P, _P, _P, _SZ, _P]),
    "fa3_qparams": (_I, [_P, _P, _P, _I, _P]),
    "fa3_range_merge": (_I, [_P, _P, _I, _I, _P, _P, _P]),
    "fa3_calibrate_f32_workspace_size": (_SZ, [_I]),
    "fa3_calibrate_perhead_f32": (_I, [_P, _I64, _I, _I64, _I64, _I64, _D, _P, _P, _P, _SZ, _P, _P]),
    "fa3_qparams_channel": (_I, [_P, _P, _I, _I, _P, _P, _P]),
    "fa3_calibrate_perchannel": (_I, [_P, _I64, _I, _I64, _I, _I64, _I64, _I64, _D, _P, _P, _P]),
    "fa3_quantize_append_channel": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "fa3_quantize_append": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P]),
    "fa3_mla_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "fa3_decode_attn_mla": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P]),
    "fa3_gqa_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "fa3_decode_attn_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P]),
    "fa3_decode_attn_gqa_channel": (_I, [_P] * 11 + [_I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P]),
    "fa3_prefill_attn_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P]),
    "fa3_quantize_append_paged": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P]),
    "fa3_decode_attn_mla_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _SZ,
                                       _P, _P]),
    "fa3_decode_attn_gqa_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P,
                                       _SZ, _P, _P]),
}


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libfa3.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libfa3.so is not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise FA3Error(fn, status)


def _need(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor of dtype {dtype}")


def _need_contig(t: torch.Tensor, dtype, name: str):
    _need(t, dtype, name)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# Cached scratch buffers, one per (call kind, device, stream), at most
# _WS_PER_KIND streams per (call kind, device): the least recently used entry is
# dropped when another stream needs one.  Callers that manage memory themselves
# pass workspace= explicitly and the cache is never touched.
_ws_cache: "OrderedDict" = OrderedDict()
_WS_PER_KIND = 4


def _ws_key(key, device, stream=None):
    dev = device.index if device.index is not None else torch.cuda.current_device()
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return (key, dev, s.cuda_stream), s


def _workspace(key, nbytes: int, device, zero: bool = False, stream=None) -> Optional[torch.Tensor]:
    """A cached scratch buffer per (call kind, device, stream): calls that share a
    workspace must not overlap, and calls on one stream never do.  It is allocated
    (and zeroed) on that stream, so its first use is ordered after the fill."""
    if nbytes == 0:
        return None
    k, s = _ws_key(key, device, stream)
    ws = _ws_cache.get(k)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(s):
            ws = (torch.zeros if zero else torch.empty)(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[k] = ws
        same = [c for c in _ws_cache if c[:2] == k[:2]]
        for old in same[:-_WS_PER_KIND]:
            if old != k:
                del _ws_cache[old]
    _ws_cache.move_to_end(k)
    return ws


def _forget_workspace(key, device, stream=None) -> None:
    _ws_cache.pop(_ws_key(key, device, stream)[0], None)


# --------------------------------------------------------------------- calls
def set_kernel_timing(start: Optional["torch.cuda.Event"], stop: Optional["torch.cuda.Event"]):
    """fa3_set_kernel_timing: later decode / calibration calls record these events
    around their main kernel (None, None turns it off).  The events must have been
    recorded once, so that their CUDA handles exist."""
    a = None if start is None else ctypes.c_void_p(start.cuda_event)
    b = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    _check("fa3_set_kernel_timing", lib().fa3_set_kernel_timing(a, b))


def calibrate_workspace_size(H: int) -> int:
    return int(lib().fa3_calibrate_workspace_size(H))


def calibrate_perhead(x: torch.Tensor, ratio: float, min_io: torch.Tensor, max_io: torch.Tensor,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Per-head Recall-Window calibration of one batch; updates min_io/max_io in place.

    x: bf16 (B, H, S, D) with (S, D) contiguous, or (H, N) with N contiguous.
    """
    _need(x, torch.bfloat16, "x")
    _need_contig(min_io, torch.float32, "min_io")
    _need_contig(max_io, torch.float32, "max_io")
    if x.dim() == 4:
        B, H, S, D = x.shape
        if x.stride(3) != 1 or x.stride(2) != D:
            raise ValueError("x must have contiguous (S, D) planes")
        L, sb, sh = S * D, x.stride(0), x.stride(1)
    elif x.dim() == 2:
        H, L = x.shape
        if x.stride(1) != 1:
            raise ValueError("x rows must be contiguous")
        B, sb, sh = 1, 0, x.stride(0)
    else:
        raise ValueError("x must be (B, H, S, D) or (H, N)")
    if min_io.numel() != H or max_io.numel() != H:
        raise ValueError("min_io/max_io must hold H values")
    nbytes = calibrate_workspace_size(H)
    cached = workspace is None
    if cached:
        workspace = _workspace("calib", nbytes, x.device, zero=True, stream=stream)
    st = lib().fa3_calibrate_perhead(_ptr(x), B, H, L, sb, sh, float(ratio), _ptr(min_io), _ptr(max_io),
                                     _ptr(workspace), workspace.numel(), _stream(stream))
    if st != 0 and cached:
        # The key counts may not have been cleared: never hand this buffer out again.
        _forget_workspace("calib", x.device, stream)
    _check("fa3_calibrate_perhead", st)


def calibrate_perhead_f32(x: torch.Tensor, ratio: float, min_io: torch.Tensor, max_io: torch.Tensor,
                          workspace: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """Per-head Recall-Window calibration of float32 activations, (B, H, S, D) with
    (S, D) contiguous or (H, N); updates min_io / max_io in place."""
    _need(x, torch.float32, "x")
    _need_contig(min_io, torch.float32, "min_io")
    _need_contig(max_io, torch.float32, "max_io")
    if x.dim() == 4:
        B, H, S, D = x.shape
        if x.stride(3) != 1 or x.stride(2) != D:
            raise ValueError("x must have contiguous (S, D) planes")
        L, sb, sh = S * D, x.stride(0), x.stride(1)
    elif x.dim() == 2:
        H, L = x.shape
        if x.stride(1) != 1:
            raise ValueError("x rows must be contiguous")
        B, sb, sh = 1, 0, x.stride(0)
    else:
        raise ValueError("x must be (B, H, S, D) or (H, N)")
    if min_io.numel() != H or max_io.numel() != H:
        raise ValueError("min_io/max_io must hold H values")
    nbytes = int(lib().fa3_calibrate_f32_workspace_size(H))
    cached = workspace is None
    if cached:
        workspace = _workspace("calib_f32", nbytes, x.device, zero=True, stream=stream)
    st = lib().fa3_calibrate_perhead_f32(_ptr(x), B, H, L, sb, sh, float(ratio), _ptr(min_io), _ptr(max_io),
                                         _ptr(workspace), workspace.numel(), _ptr(dev_err), _stream(stream))
    if st != 0 and cached:
        _forget_workspace("calib_f32", x.device, stream)
    _check("fa3_calibrate_perhead_f32", st)


def range_merge(mins: torch.Tensor, maxs: torch.Tensor, min_io: torch.Tensor, max_io: torch.Tensor,
                stream=None) -> None:
    """Folds R ranges mins/maxs [R][H] into the running range min_io/max_io [H] (in place)."""
    _need_contig(mins, torch.float32, "mins")
    _need_contig(maxs, torch.float32, "maxs")
    _need_contig(min_io, torch.float32, "min_io")
    _need_contig(max_io, torch.float32, "max_io")
    H = min_io.numel()
    if mins.dim() != 2 or mins.shape != maxs.shape or mins.shape[1] != H or max_io.numel() != H:
        raise ValueError("mins/maxs must be [R][H] with H = min_io.numel()")
    st = lib().fa3_range_merge(_ptr(mins), _ptr(maxs), mins.shape[0], H, _ptr(min_io), _ptr(max_io),
                               _stream(stream))
    _check("fa3_range_merge", st)


def calibrate_perhead_sharded(batches, ratio: float, min_io: torch.Tensor, max_io: torch.Tensor,
                              group=None, stream=None) -> None:
    """Recall-Window calibration with the batches sharded over the ranks of a
    torch.distributed group: each rank calibrates its own batches into a local
    range (fa3_calibrate_perhead), the ranks all-gather their [H] ranges (the one
    exchange step), and every rank folds them into min_io/max_io
    (fa3_range_merge).  Step 3 is associative, so the result is bit-identical to
    one process accumulating every batch in any order."""
    import torch.distributed as dist
    H = min_io.numel()
    dev = min_io.device
    loc_mn = torch.full((H,), float("inf"), dtype=torch.float32, device=dev)
    loc_mx = torch.full((H,), float("-inf"), dtype=torch.float32, device=dev)
    for x in batches:
        calibrate_perhead(x, ratio, loc_mn, loc_mx, stream=stream)
    world = dist.get_world_size(group)
    mins = torch.empty(world, H, dtype=torch.float32, device=dev)
    maxs = torch.empty(world, H, dtype=torch.float32, device=dev)
    ctx = torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()
    with ctx:                                   # the collective is ordered on the calls' stream
        dist.all_gather(list(mins.unbind(0)), loc_mn, group=group)    # rows of mins / maxs
        dist.all_gather(list(maxs.unbind(0)), loc_mx, group=group)
    range_merge(mins, maxs, min_io, max_io, stream=stream)


def qparams(min_v: torch.Tensor, max_v: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None):
    _need_contig(min_v, torch.float32, "min")
    _need_contig(max_v, torch.float32, "max")
    H = min_v.numel()
    if out is None:
        out = torch.empty(H, dtype=torch.float32, device=min_v.device)
    st = lib().fa3_qparams(_ptr(min_v), _ptr(max_v), _ptr(out), H, _stream(stream))
    _check("fa3_qparams", st)
    return out


def calibrate_perchannel(x: torch.Tensor, ratio: float, min_io: torch.Tensor, max_io: torch.Tensor,
                         stream=None) -> None:
    """Recall-Window calibration per (head, channel) of one batch x bf16 (B, H, S, D)
    (D contiguous); updates min_io / max_io [H][D] in place."""
    _need(x, torch.bfloat16, "x")
    _need_contig(min_io, torch.float32, "min_io")
    _need_contig(max_io, torch.float32, "max_io")
    if x.dim() != 4 or x.stride(3) != 1:
        raise ValueError("x must be (B, H, S, D) with D contiguous")
    B, H, S, D = x.shape
    if min_io.numel() != H * D or max_io.numel() != H * D:
        raise ValueError("min_io / max_io must hold H * D values")
    st = lib().fa3_calibrate_perchannel(_ptr(x), B, H, S, D, x.stride(0), x.stride(1), x.stride(2), float(ratio),
                                        _ptr(min_io), _ptr(max_io), _stream(stream))
    _check("fa3_calibrate_perchannel", st)


def qparams_channel(min_v: torch.Tensor, max_v: torch.Tensor, asymmetric: bool, stream=None):
    """Per-(head, channel) scale and offset from per-channel ranges [H][D]; returns (scale, offset)."""
    _need_contig(min_v, torch.float32, "min")
    _need_contig(max_v, torch.float32, "max")
    if min_v.shape != max_v.shape:
        raise ValueError("min and max must have the same shape")
    scale = torch.empty_like(min_v)
    offset = torch.empty_like(min_v)
    st = lib().fa3_qparams_channel(_ptr(min_v), _ptr(max_v), min_v.numel(), int(bool(asymmetric)), _ptr(scale),
                                   _ptr(offset), _stream(stream))
    _check("fa3_qparams_channel", st)
    return scale, offset


def quantize_append_channel(kv: torch.Tensor, scale: torch.Tensor, offset: Optional[torch.Tensor], asymmetric: bool,
                            cache: torch.Tensor, pos: torch.Tensor, dev_err: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    """kv bf16 [B][T_new][H][D] -> cache int8 [B][T_max][H][D] at pos[b], per-channel scale/offset [H][D]."""
    _need_contig(kv, torch.bfloat16, "kv")
    _need_contig(scale, torch.float32, "scale")
    if asymmetric:
        _need_contig(offset, torch.float32, "offset")
    _need_contig(cache, torch.int8, "cache")
    _need_contig(pos, torch.int32, "pos")
    B, T_new, H, D = kv.shape
    if cache.dim() != 4 or cache.shape[0] != B or cache.shape[2] != H or cache.shape[3] != D:
        raise ValueError("cache must be [B][T_max][H][D]")
    if scale.numel() != H * D or (asymmetric and offset.numel() != H * D):
        raise ValueError("scale / offset must hold H * D values")
    st = lib().fa3_quantize_append_channel(_ptr(kv), _ptr(scale), _ptr(offset) if asymmetric else None,
                                           int(bool(asymmetric)), _ptr(cache), _ptr(pos), B, T_new, H, D,
                                           cache.shape[1], _ptr(dev_err), _stream(stream))
    _check("fa3_quantize_append_channel", st)


def quantize_append(kv: torch.Tensor, scale: torch.Tensor, cache: torch.Tensor, pos: torch.Tensor,
                    rope_src: Optional[torch.Tensor] = None, rope_cache: Optional[torch.Tensor] = None,
                    dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """kv bf16 [B][T_new][H][D] -> cache int8 [B][T_max][H][D] at pos[b]."""
    _need_contig(kv, torch.bfloat16, "kv")
    _need_contig(scale, torch.float32, "scale")
    _need_contig(cache, torch.int8, "cache")
    _need_contig(pos, torch.int32, "pos")
    B, T_new, H, D = kv.shape
    if cache.dim() != 4 or cache.shape[0] != B or cache.shape[2] != H or cache.shape[3] != D:
        raise ValueError("cache must be [B][T_max][H][D]")
    Dr = 0
    if rope_src is not None:
        _need_contig(rope_src, torch.bfloat16, "rope_src")
        _need_contig(rope_cache, torch.bfloat16, "rope_cache")
        Dr = rope_src.shape[-1]
    st = lib().fa3_quantize_append(_ptr(kv), _ptr(scale), _ptr(cache), _ptr(pos), B, T_new, H, D, cache.shape[1],
                                   _ptr(rope_src), _ptr(rope_cache), Dr, _ptr(dev_err), _stream(stream))
    _check("fa3_quantize_append", st)


def mla_workspace_size(B: int, H: int, Dl: int, T_max: int) -> int:
    return int(lib().fa3_mla_workspace_size(B, H, Dl, T_max))


def decode_attn_mla(q: torch.Tensor, ckv: torch.Tensor, krope: torch.Tensor, q_scale: torch.Tensor,
                    kv_scale: torch.Tensor, lens: torch.Tensor, softmax_scale: float,
                    out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Absorbed-MLA decode: q bf16 [B][H][Dl+Dr], ckv int8 [B][T_max][Dl], krope bf16 [B][T_max][Dr]."""
    _need_contig(q, torch.bfloat16, "q")
    _need_contig(ckv, torch.int8, "ckv")
    _need_contig(krope, torch.bfloat16, "krope")
    _need_contig(q_scale, torch.float32, "q_scale")
    _need_contig(kv_scale, torch.float32, "kv_scale")
    _need_contig(lens, torch.int32, "lens")
    B, H, Dqk = q.shape
    T_max, Dl = ckv.shape[1], ckv.shape[2]
    Dr = krope.shape[2]
    if Dqk != Dl + Dr:
        raise ValueError("q last dim must be Dl + Dr")
    if out is None:
        out = torch.empty(B, H, Dl, dtype=torch.float32, device=q.device)
    nbytes = mla_workspace_size(B, H, Dl, T_max)
    if workspace is None:
        workspace = _workspace("mla", nbytes, q.device, stream=stream)
    st = lib().fa3_decode_attn_mla(_ptr(q), _ptr(ckv), _ptr(krope), _ptr(q_scale), _ptr(kv_scale), _ptr(lens),
                                   _ptr(out), B, H, Dl, Dr, T_max, float(softmax_scale), _ptr(workspace),
                                   0 if workspace is None else workspace.numel(), _ptr(dev_err), _stream(stream))
    _check("fa3_decode_attn_mla", st)
    return out


def gqa_workspace_size(B: int, Hq: int, Hkv: int, D: int, T_max: int) -> int:
    return int(lib().fa3_gqa_workspace_size(B, Hq, Hkv, D, T_max))


def decode_attn_gqa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_scale: torch.Tensor,
                    k_scale: torch.Tensor, v_scale: torch.Tensor, lens: torch.Tensor, softmax_scale: float,
                    out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """GQA decode: q int8 [B][Hq][D], k/v int8 [B][T_max][Hkv][D] -> bf16 [B][Hq][D]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need_contig(t, torch.int8, n)
    for t, n in ((q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        _need_contig(t, torch.float32, n)
    _need_contig(lens, torch.int32, "lens")
    B, Hq, D = q.shape
    T_max, Hkv = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=q.device)
    nbytes = gqa_workspace_size(B, Hq, Hkv, D, T_max)
    if workspace is None:
        workspace = _workspace("gqa", nbytes, q.device, stream=stream)
    st = lib().fa3_decode_attn_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(lens), _ptr(out), B, Hq, Hkv, D, T_max, float(softmax_scale),
                                   _ptr(workspace), 0 if workspace is None else workspace.numel(),
                                   _ptr(dev_err), _stream(stream))
    _check("fa3_decode_attn_gqa", st)
    return out


def decode_attn_gqa_channel(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_scale: torch.Tensor,
                            q_offset: torch.Tensor, k_scale: torch.Tensor, k_offset: torch.Tensor,
                            v_scale: torch.Tensor, v_offset: torch.Tensor, lens: torch.Tensor, softmax_scale: float,
                            out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """GQA decode with per-channel scales / offsets ([heads][D] each): q int8 [B][Hq][D],
    k/v int8 [B][T_max][Hkv][D] -> bf16 [B][Hq][D]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need_contig(t, torch.int8, n)
    for t, n in ((q_scale, "q_scale"), (q_offset, "q_offset"), (k_scale, "k_scale"), (k_offset, "k_offset"),
                 (v_scale, "v_scale"), (v_offset, "v_offset")):
        _need_contig(t, torch.float32, n)
    _need_contig(lens, torch.int32, "lens")
    B, Hq, D = q.shape
    T_max, Hkv = k.shape[1], k.shape[2]
    if q_scale.numel() != Hq * D or k_scale.numel() != Hkv * D or v_scale.numel() != Hkv * D:
        raise ValueError("per-channel parameters must be [heads][D]")
    if out is None:
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=q.device)
    nbytes = gqa_workspace_size(B, Hq, Hkv, D, T_max)
    if workspace is None:
        workspace = _workspace("gqa", nbytes, q.device, stream=stream)
    st = lib().fa3_decode_attn_gqa_channel(_ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(q_offset), _ptr(k_scale),
                                           _ptr(k_offset), _ptr(v_scale), _ptr(v_offset), _ptr(lens), _ptr(out), B,
                                           Hq, Hkv, D, T_max, float(softmax_scale), _ptr(workspace),
                                           0 if workspace is None else workspace.numel(), _ptr(dev_err),
                                           _stream(stream))
    _check("fa3_decode_attn_gqa_channel", st)
    return out


def prefill_attn_gqa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_scale: torch.Tensor,
                     k_scale: torch.Tensor, v_scale: torch.Tensor, q_lens: torch.Tensor, kv_lens: torch.Tensor,
                     softmax_scale: float, out: Optional[torch.Tensor] = None,
                     dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal prefill: q int8 [B][S][Hq][D], k/v int8 [B][T][Hkv][D] -> bf16 [B][S][Hq][D].

    Rows i >= q_lens[b] of ``out`` are left untouched (zero-filled when ``out`` is
    allocated here)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need_contig(t, torch.int8, n)
    for t, n in ((q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        _need_contig(t, torch.float32, n)
    _need_contig(q_lens, torch.int32, "q_lens")
    _need_contig(kv_lens, torch.int32, "kv_lens")
    B, S, Hq, D = q.shape
    T, Hkv = k.shape[1], k.shape[2]
    if out is None:
        out = torch.zeros(B, S, Hq, D, dtype=torch.bfloat16, device=q.device)
    _need_contig(out, torch.bfloat16, "out")
    st = lib().fa3_prefill_attn_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                    _ptr(q_lens), _ptr(kv_lens), _ptr(out), B, S, T, Hq, Hkv, D,
                                    float(softmax_scale), _ptr(dev_err), _stream(stream))
    _check("fa3_prefill_attn_gqa", st)
    return out


# ------------------------------------------------------------- paged cache
def _block_table(block_table: torch.Tensor, B: int) -> int:
    _need_contig(block_table, torch.int32, "block_table")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B][max_pages]")
    return block_table.shape[1]


def quantize_append_paged(kv: torch.Tensor, scale: torch.Tensor, cache: torch.Tensor, block_table: torch.Tensor,
                          pos: torch.Tensor, rope_src: Optional[torch.Tensor] = None,
                          rope_cache: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """kv bf16 [B][T_new][H][D] -> page pool int8 [num_pages][page_size][H][D] at pos[b]."""
    _need_contig(kv, torch.bfloat16, "kv")
    _need_contig(scale, torch.float32, "scale")
    _need_contig(cache, torch.int8, "cache")
    _need_contig(pos, torch.int32, "pos")
    B, T_new, H, D = kv.shape
    if cache.dim() != 4 or cache.shape[2] != H or cache.shape[3] != D:
        raise ValueError("cache must be [num_pages][page_size][H][D]")
    num_pages, page_size = cache.shape[0], cache.shape[1]
    max_pages = _block_table(block_table, B)
    Dr = 0
    if rope_src is not None:
        _need_contig(rope_src, torch.bfloat16, "rope_src")
        _need_contig(rope_cache, torch.bfloat16, "rope_cache")
        Dr = rope_src.shape[-1]
    st = lib().fa3_quantize_append_paged(_ptr(kv), _ptr(scale), _ptr(cache), _ptr(block_table), _ptr(pos), B, T_new,
                                         H, D, num_pages, page_size, max_pages, _ptr(rope_src), _ptr(rope_cache), Dr,
                                         _ptr(dev_err), _stream(stream))
    _check("fa3_quantize_append_paged", st)


def decode_attn_mla_paged(q: torch.Tensor, ckv: torch.Tensor, krope: torch.Tensor, q_scale: torch.Tensor,
                          kv_scale: torch.Tensor, lens: torch.Tensor, block_table: torch.Tensor, softmax_scale: float,
                          out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Absorbed-MLA decode over page pools: ckv int8 [num_pages][page_size][Dl], krope bf16 [...][Dr]."""
    _need_contig(q, torch.bfloat16, "q")
    _need_contig(ckv, torch.int8, "ckv")
    _need_contig(krope, torch.bfloat16, "krope")
    _need_contig(q_scale, torch.float32, "q_scale")
    _need_contig(kv_scale, torch.float32, "kv_scale")
    _need_contig(lens, torch.int32, "lens")
    B, H, Dqk = q.shape
    num_pages, page_size, Dl = ckv.shape
    Dr = krope.shape[2]
    if Dqk != Dl + Dr:
        raise ValueError("q last dim must be Dl + Dr")
    max_pages = _block_table(block_table, B)
    if out is None:
        out = torch.empty(B, H, Dl, dtype=torch.float32, device=q.device)
    nbytes = mla_workspace_size(B, H, Dl, max_pages * page_size)
    if workspace is None:
        workspace = _workspace("mla", nbytes, q.device, stream=stream)
    st = lib().fa3_decode_attn_mla_paged(_ptr(q), _ptr(ckv), _ptr(krope), _ptr(q_scale), _ptr(kv_scale), _ptr(lens),
                                         _ptr(block_table), _ptr(out), B, H, Dl, Dr, num_pages, page_size, max_pages,
                                         float(softmax_scale), _ptr(workspace),
                                         0 if workspace is None else workspace.numel(), _ptr(dev_err),
                                         _stream(stream))
    _check("fa3_decode_attn_mla_paged", st)
    return out


def decode_attn_gqa_paged(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_scale: torch.Tensor,
                          k_scale: torch.Tensor, v_scale: torch.Tensor, lens: torch.Tensor, block_table: torch.Tensor,
                          softmax_scale: float, out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """GQA decode over page pools: k/v int8 [num_pages][page_size][Hkv][D] -> bf16 [B][Hq][D]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need_contig(t, torch.int8, n)
    for t, n in ((q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        _need_contig(t, torch.float32, n)
    _need_contig(lens, torch.int32, "lens")
    B, Hq, D = q.shape
    num_pages, page_size, Hkv = k.shape[0], k.shape[1], k.shape[2]
    max_pages = _block_table(block_table, B)
    if out is None:
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=q.device)
    nbytes = gqa_workspace_size(B, Hq, Hkv, D, max_pages * page_size)
    if workspace is None:
        workspace = _workspace("gqa", nbytes, q.device, stream=stream)
    st = lib().fa3_decode_attn_gqa_paged(_ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                         _ptr(lens), _ptr(block_table), _ptr(out), B, Hq, Hkv, D, num_pages,
                                         page_size, max_pages, float(softmax_scale), _ptr(workspace),
                                         0 if workspace is None else workspace.numel(), _ptr(dev_err),
                                         _stream(stream))
    _check("fa3_decode_attn_gqa_paged", st)
    return out
