"""audio_dit_gb300 -- GB300 (sm_103a) NVFP4 linear path of a joint video/audio DiT.

Thin Python binding over the C ABI in ``include/h3fp4.h`` (``libh3fp4.so``):
the functions below carry the C names and only marshal arguments -- every
step of the path (modulation, amax, block scales, E2M1 packing, block-scaled
GEMM, bias/gate/residual epilogue) runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.  There is no CPU or eager
fallback: if the library is missing or the device is not sm_103 the calls
raise.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

__all__ = [
    "H3FP4Error", "PROLOGUE_MOD", "EPI_BIAS", "EPI_GATE_RESID", "GSCALE_GIVEN", "A_PREQUANT",
    "EPI_SWIGLU", "EPI_AMAX", "FUSED_QUANT", "h3fp4_ws_out_amax", "h3fp4_selftest_pack_timeout",
    "MAX_SEGMENTS", "library_path", "load_library", "h3fp4_codes_bytes", "h3fp4_sf_bytes",
    "h3fp4_workspace_bytes", "h3fp4_quantize_weight", "h3fp4_quantize_act", "h3fp4_linear",
    "h3fp4_check", "h3fp4_act_amax", "h3fp4_gscale_from_amax", "h3fp4_selftest_timeout", "h3fp4_measure_fp4_peak", "h3fp4_measure_fp4_pair_peak", "h3fp4_measure_fp4_form", "MMA_FORMS", "h3fp4_quantize_act_noalloc",
    "h3fp4_linear_swiglu_nvfp4", "h3fp4_set_wait_limit_ns", "h3fp4_status_string", "alloc_nvfp4", "alloc_workspace",
]

PROLOGUE_MOD = 1
EPI_BIAS = 2
EPI_GATE_RESID = 4
GSCALE_GIVEN = 16
A_PREQUANT = 32
EPI_SWIGLU = 64
EPI_AMAX = 128
FUSED_QUANT = 256
MAX_SEGMENTS = 8

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


class H3FP4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: h3fp4 status {status} ({h3fp4_status_string(status)})")


def library_path() -> str:
    return os.path.join(_HERE, "_build", "libh3fp4.so")


def load_library():
    """Load libh3fp4.so (build it first with ``python -m audio_dit_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"libh3fp4.so not built ({path}); run `python -m audio_dit_gb300.build`")
    L = C.CDLL(path)
    i64, vp, i32, sz = C.c_int64, C.c_void_p, C.c_int, C.c_size_t
    sig = {
        "h3fp4_codes_bytes": (sz, [i64, i64]),
        "h3fp4_sf_bytes": (sz, [i64, i64]),
        "h3fp4_workspace_bytes": (sz, [i64, i64, i64, i32]),
        "h3fp4_quantize_weight": (i32, [vp, i64, i64, vp, vp, vp, vp, vp]),
        "h3fp4_quantize_act": (i32, [vp, i64, i64, vp, vp, vp, i32, vp, vp, vp, i32, vp, vp]),
        "h3fp4_linear": (i32, [vp, vp, vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp,
                               i32, vp, vp]),
        "h3fp4_act_amax": (i32, [vp, i64, i64, vp, vp, vp, i32, vp, i32, vp, vp]),
        "h3fp4_linear_swiglu_nvfp4": (i32, [vp, vp, vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp,
                                            i32, vp, vp]),
        "h3fp4_gscale_from_amax": (i32, [vp, vp, vp]),
        "h3fp4_ws_out_amax": (vp, [vp]),
        "h3fp4_selftest_timeout": (i32, [vp, C.c_uint64, vp]),
        "h3fp4_selftest_pack_timeout": (i32, [vp, vp, vp, C.c_uint64, vp]),
        "h3fp4_measure_fp4_peak": (i32, [i32, vp, vp]),
        "h3fp4_measure_fp4_pair_peak": (i32, [i32, vp, vp]),
        "h3fp4_measure_fp4_form": (i32, [i32, i32, vp, vp]),
        "h3fp4_quantize_act_noalloc": (i32, [vp, i64, i64, vp, vp, vp, i32, vp, vp, vp, i32, vp]),
        "h3fp4_check": (i32, [vp, vp]),
        "h3fp4_set_wait_limit_ns": (None, [C.c_uint64]),
        "h3fp4_status_string": (C.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


# ------------------------------------------------------------------ marshalling helpers

def _ptr(t: Optional[torch.Tensor], what: str, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _segs(seg_off: Optional[Sequence[int]]):
    if seg_off is None:
        return None, 1, None
    arr = (C.c_int64 * len(seg_off))(*[int(v) for v in seg_off])
    return C.cast(arr, C.c_void_p), len(seg_off) - 1, arr


def _check(status: int, what: str):
    if status != 0:
        raise H3FP4Error(status, what)


# ------------------------------------------------------------------ C-ABI functions

def h3fp4_status_string(status: int) -> str:
    return load_library().h3fp4_status_string(status).decode()


def h3fp4_codes_bytes(rows: int, K: int) -> int:
    return int(load_library().h3fp4_codes_bytes(rows, K))


def h3fp4_sf_bytes(rows: int, K: int) -> int:
    return int(load_library().h3fp4_sf_bytes(rows, K))


def h3fp4_workspace_bytes(M: int, N: int, K: int, flags: int = 0) -> int:
    return int(load_library().h3fp4_workspace_bytes(M, N, K, flags))


def h3fp4_set_wait_limit_ns(ns: int) -> None:
    load_library().h3fp4_set_wait_limit_ns(int(ns))


def h3fp4_quantize_weight(w: torch.Tensor, codes: torch.Tensor, sf: torch.Tensor, gscale: torch.Tensor,
                          ws: torch.Tensor, stream=None) -> None:
    N, K = w.shape
    _check(load_library().h3fp4_quantize_weight(
        _ptr(w, "w", torch.bfloat16), N, K, _ptr(codes, "codes", torch.uint8), _ptr(sf, "sf", torch.uint8),
        _ptr(gscale, "gscale", torch.float32), _ptr(ws, "ws", torch.uint8), _stream(stream)),
        "h3fp4_quantize_weight")


def h3fp4_quantize_act(x: torch.Tensor, codes: torch.Tensor, sf: torch.Tensor, gscale: torch.Tensor,
                       ws: torch.Tensor, shift: Optional[torch.Tensor] = None,
                       scale: Optional[torch.Tensor] = None, seg_off: Optional[Sequence[int]] = None,
                       gscale_given: bool = False, stream=None) -> None:
    M, K = x.shape
    flags = (PROLOGUE_MOD if shift is not None else 0) | (GSCALE_GIVEN if gscale_given else 0)
    sp, nseg, _keep = _segs(seg_off)
    _check(load_library().h3fp4_quantize_act(
        _ptr(x, "x", torch.bfloat16), M, K, _ptr(shift, "shift", torch.float32),
        _ptr(scale, "scale", torch.float32), sp, nseg, _ptr(codes, "codes", torch.uint8),
        _ptr(sf, "sf", torch.uint8), _ptr(gscale, "gscale", torch.float32), flags,
        _ptr(ws, "ws", torch.uint8), _stream(stream)), "h3fp4_quantize_act")


def h3fp4_linear(x: torch.Tensor, w_codes: torch.Tensor, w_sf: torch.Tensor, w_gscale: torch.Tensor,
                 out: torch.Tensor, ws: torch.Tensor, *, K: Optional[int] = None,
                 a_sf: Optional[torch.Tensor] = None, a_gscale: Optional[torch.Tensor] = None,
                 shift: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None,
                 gate: Optional[torch.Tensor] = None, resid: Optional[torch.Tensor] = None,
                 bias: Optional[torch.Tensor] = None, seg_off: Optional[Sequence[int]] = None,
                 gscale_given: bool = False, swiglu: bool = False, out_amax: bool = False,
                 fused: bool = False, stream=None) -> None:
    """out = [R + g*](alpha * NVFP4(prologue(x)) . W^T [+ b]).

    ``x`` is bf16 [M, K]; or uint8 codes [M, K/2] together with ``a_sf`` and
    ``a_gscale`` (pre-quantised activation).  ``swiglu``: out is [M, N/2] =
    bf16(silu(g) * u) over the weight's [gate 128 | up 128] row groups.
    ``out_amax``: also leave max|out| at :func:`h3fp4_ws_out_amax` (ws).
    ``fused``: the GEMM kernel quantises x itself (H3FP4_FUSED_QUANT).
    """
    prequant = x.dtype == torch.uint8
    M = x.shape[0]
    K = x.shape[1] * (2 if prequant else 1)
    N = out.shape[1] * (2 if swiglu else 1)
    flags = ((A_PREQUANT if prequant else 0) | (PROLOGUE_MOD if shift is not None else 0)
             | (EPI_BIAS if bias is not None else 0) | (EPI_GATE_RESID if gate is not None else 0)
             | (GSCALE_GIVEN if gscale_given else 0) | (EPI_SWIGLU if swiglu else 0)
             | (EPI_AMAX if out_amax else 0) | (FUSED_QUANT if fused else 0))
    sp, nseg, _keep = _segs(seg_off)
    _check(load_library().h3fp4_linear(
        _ptr(x, "x"), _ptr(a_sf, "a_sf", torch.uint8), _ptr(a_gscale, "a_gscale", torch.float32), M, N, K,
        _ptr(w_codes, "w_codes", torch.uint8), _ptr(w_sf, "w_sf", torch.uint8),
        _ptr(w_gscale, "w_gscale", torch.float32), _ptr(shift, "shift", torch.float32),
        _ptr(scale, "scale", torch.float32), _ptr(gate, "gate", torch.float32), sp, nseg,
        _ptr(bias, "bias", torch.bfloat16), _ptr(resid, "resid", torch.bfloat16),
        _ptr(out, "out", torch.bfloat16), flags, _ptr(ws, "ws", torch.uint8), _stream(stream)),
        "h3fp4_linear")


def h3fp4_linear_swiglu_nvfp4(x: torch.Tensor, w_codes: torch.Tensor, w_sf: torch.Tensor, w_gscale: torch.Tensor,
                              h_codes: torch.Tensor, h_sf: torch.Tensor, h_gscale: torch.Tensor, ws: torch.Tensor, *,
                              a_sf: Optional[torch.Tensor] = None, a_gscale: Optional[torch.Tensor] = None,
                              shift: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None,
                              bias: Optional[torch.Tensor] = None, seg_off: Optional[Sequence[int]] = None,
                              gscale_given: bool = False, stream=None) -> None:
    """FC1 with the SwiGLU producer writing h = bf16(silu(g) * u) as NVFP4:
    ``h_codes`` uint8 [M, N/4], ``h_sf`` (h3fp4_sf_bytes(M, N/2)) under the
    given global scale ``h_gscale`` (device fp32 [1], an input)."""
    prequant = x.dtype == torch.uint8
    M = x.shape[0]
    K = x.shape[1] * (2 if prequant else 1)
    N = h_codes.shape[1] * 4
    flags = ((A_PREQUANT if prequant else 0) | (PROLOGUE_MOD if shift is not None else 0)
             | (EPI_BIAS if bias is not None else 0) | (GSCALE_GIVEN if gscale_given else 0))
    sp, nseg, _keep = _segs(seg_off)
    _check(load_library().h3fp4_linear_swiglu_nvfp4(
        _ptr(x, "x"), _ptr(a_sf, "a_sf", torch.uint8), _ptr(a_gscale, "a_gscale", torch.float32), M, N, K,
        _ptr(w_codes, "w_codes", torch.uint8), _ptr(w_sf, "w_sf", torch.uint8),
        _ptr(w_gscale, "w_gscale", torch.float32), _ptr(shift, "shift", torch.float32),
        _ptr(scale, "scale", torch.float32), sp, nseg, _ptr(bias, "bias", torch.bfloat16),
        _ptr(h_gscale, "h_gscale", torch.float32), _ptr(h_codes, "h_codes", torch.uint8),
        _ptr(h_sf, "h_sf", torch.uint8), flags, _ptr(ws, "ws", torch.uint8), _stream(stream)),
        "h3fp4_linear_swiglu_nvfp4")


def h3fp4_quantize_act_noalloc(x: torch.Tensor, codes: torch.Tensor, sf: torch.Tensor, gscale: torch.Tensor,
                               shift: Optional[torch.Tensor] = None, scale: Optional[torch.Tensor] = None,
                               seg_off: Optional[Sequence[int]] = None, gscale_given: bool = False,
                               stream=None) -> None:
    """h3fp4_quantize_act without a workspace, for callers that may not allocate
    device memory; its scratch is a static device array shared by all calls
    (serialise calls that could overlap on the GPU)."""
    M, K = x.shape
    flags = (PROLOGUE_MOD if shift is not None else 0) | (GSCALE_GIVEN if gscale_given else 0)
    sp, nseg, _keep = _segs(seg_off)
    _check(load_library().h3fp4_quantize_act_noalloc(
        _ptr(x, "x", torch.bfloat16), M, K, _ptr(shift, "shift", torch.float32),
        _ptr(scale, "scale", torch.float32), sp, nseg, _ptr(codes, "codes", torch.uint8),
        _ptr(sf, "sf", torch.uint8), _ptr(gscale, "gscale", torch.float32), flags, _stream(stream)),
        "h3fp4_quantize_act_noalloc")


def h3fp4_act_amax(x: torch.Tensor, amax: torch.Tensor, ws: torch.Tensor, shift: Optional[torch.Tensor] = None,
                   scale: Optional[torch.Tensor] = None, seg_off: Optional[Sequence[int]] = None,
                   stream=None) -> None:
    """amax of this call's (modulated) rows into ``amax`` (device fp32 [1])."""
    M, K = x.shape
    sp, nseg, _keep = _segs(seg_off)
    _check(load_library().h3fp4_act_amax(
        _ptr(x, "x", torch.bfloat16), M, K, _ptr(shift, "shift", torch.float32),
        _ptr(scale, "scale", torch.float32), sp, nseg, _ptr(amax, "amax", torch.float32),
        PROLOGUE_MOD if shift is not None else 0, _ptr(ws, "ws", torch.uint8), _stream(stream)),
        "h3fp4_act_amax")


def h3fp4_ws_out_amax(ws: torch.Tensor) -> torch.Tensor:
    """The fp32 [1] view of ``ws`` where an ``out_amax`` linear leaves max|out|."""
    addr = load_library().h3fp4_ws_out_amax(_ptr(ws, "ws", torch.uint8))
    off = int(addr) - ws.data_ptr()
    return ws[off:off + 4].view(torch.float32)


def h3fp4_gscale_from_amax(amax: torch.Tensor, gscale: torch.Tensor, stream=None) -> None:
    _check(load_library().h3fp4_gscale_from_amax(_ptr(amax, "amax", torch.float32),
                                                 _ptr(gscale, "gscale", torch.float32), _stream(stream)),
           "h3fp4_gscale_from_amax")


def h3fp4_selftest_timeout(ws: torch.Tensor, limit_ns: int, stream=None) -> None:
    _check(load_library().h3fp4_selftest_timeout(_ptr(ws, "ws", torch.uint8), int(limit_ns), _stream(stream)),
           "h3fp4_selftest_timeout")


def h3fp4_selftest_pack_timeout(x: torch.Tensor, a_gscale: torch.Tensor, ws: torch.Tensor, limit_ns: int,
                                stream=None) -> None:
    _check(load_library().h3fp4_selftest_pack_timeout(_ptr(x, "x", torch.bfloat16),
                                                      _ptr(a_gscale, "a_gscale", torch.float32),
                                                      _ptr(ws, "ws", torch.uint8), int(limit_ns), _stream(stream)),
           "h3fp4_selftest_pack_timeout")


def h3fp4_measure_fp4_peak(ws: torch.Tensor, iters: int = 20000) -> float:
    """Measured FP4 MMA ceiling (TFLOP/s) of the current device (synchronous)."""
    out = C.c_float(0.0)
    _check(load_library().h3fp4_measure_fp4_peak(int(iters), C.byref(out), _ptr(ws, "ws", torch.uint8)),
           "h3fp4_measure_fp4_peak")
    return float(out.value)


def h3fp4_measure_fp4_pair_peak(ws: torch.Tensor, iters: int = 20000) -> float:
    """Measured ceiling (TFLOP/s) of the paired (2-CTA) FP4 MMA the GEMM issues (synchronous)."""
    out = C.c_float(0.0)
    _check(load_library().h3fp4_measure_fp4_pair_peak(int(iters), C.byref(out), _ptr(ws, "ws", torch.uint8)),
           "h3fp4_measure_fp4_pair_peak")
    return float(out.value)


MMA_FORMS = {0: "cta_group::1 M=128 N=256 K=64, A smem", 1: "cta_group::2 M=256 N=256 K=64, A smem",
             2: "cta_group::1, A TMEM", 3: "cta_group::2, A TMEM", 4: "cta_group::1, 2 x N=128 sharing A",
             5: "cta_group::1, 2 x N=128, collector::a fill/lastuse", 6: "cta_group::2, 2 x N=128 sharing A"}


def h3fp4_measure_fp4_form(ws: torch.Tensor, form: int, iters: int = 20000) -> float:
    """Measured ceiling (TFLOP/s) of one kind::mxf4nvf4 MMA form (MMA_FORMS; synchronous)."""
    out = C.c_float(0.0)
    _check(load_library().h3fp4_measure_fp4_form(int(form), int(iters), C.byref(out), _ptr(ws, "ws", torch.uint8)),
           "h3fp4_measure_fp4_form")
    return float(out.value)


def h3fp4_check(ws: torch.Tensor, stream=None) -> None:
    """Synchronise and raise H3FP4Error if a device wait timed out."""
    _check(load_library().h3fp4_check(_ptr(ws, "ws", torch.uint8), _stream(stream)), "h3fp4_check")


# ------------------------------------------------------------------ buffer helpers (torch allocations)

def alloc_nvfp4(rows: int, K: int, device="cuda"):
    """(codes uint8 [rows, K/2], sf uint8 [sf_bytes], gscale fp32 [1]) on ``device``."""
    return (torch.empty((rows, K // 2), dtype=torch.uint8, device=device),
            torch.empty(h3fp4_sf_bytes(rows, K), dtype=torch.uint8, device=device),
            torch.empty(1, dtype=torch.float32, device=device))


def alloc_workspace(M: int, N: int, K: int, flags: int = 0, device="cuda") -> torch.Tensor:
    return torch.zeros(h3fp4_workspace_bytes(M, N, K, flags), dtype=torch.uint8, device=device)
