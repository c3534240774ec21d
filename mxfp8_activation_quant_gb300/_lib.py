"""ctypes binding of libmxq (include/mxq.h): argument marshalling only.

Every computation runs in the CUDA library; this module turns torch tensors into pointers,
sizes and the caller's current stream, and turns status codes into exceptions. If the
library has not been built (``python -c "import __graft_entry__ as g; g.build()"``) every
call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmxq.so")

SF_ROWMAJOR_U8 = 0
SF_PACKED_I32_MN = 1
SF_TILED_128X4 = 2

STATUS_NAMES = {0: "MXQ_OK", 1: "MXQ_ERR_INVALID_ARG", 2: "MXQ_ERR_UNSUPPORTED_SHAPE", 3: "MXQ_ERR_MISALIGNED",
                4: "MXQ_ERR_LAYOUT", 5: "MXQ_ERR_CUDA", 6: "MXQ_ERR_TIMEOUT"}


class MxqError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class MxTensorC(ctypes.Structure):
    """The C struct mxq_mx_tensor."""
    _fields_ = [("data", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("sf_layout", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ld", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None

P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
_MXP = ctypes.POINTER(MxTensorC)
SIGNATURES = {
    "mxq_abi_version": ([], ctypes.c_int),
    "mxq_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "mxq_last_error_string": ([], ctypes.c_char_p),
    "mxq_sf_bytes": ([I32, I64, I64], ctypes.c_size_t),
    "mxq_status_bytes": ([], ctypes.c_size_t),
    "mxq_check_status": ([P, P], ctypes.c_int),
    "mxq_selftest_wait_timeout": ([I64, P, P], ctypes.c_int),
    "mxq_selftest_hold_sms": ([I64, I64, P], ctypes.c_int),
    "mxfp8_quantize": ([P, I64, I64, I64, P, I64, P, P, P, P], ctypes.c_int),
    "rmsnorm_dual_out": ([P, P, ctypes.c_float, I64, I64, I64, P, P, P, P, P, P], ctypes.c_int),
    "mxq_workspace_bytes": ([], I64),
    "wo_a_einsum_mxfp8": ([_MXP, _MXP, I64, I32, I32, I32, P, P, P, P, P, I64, P, P], ctypes.c_int),
    "gemm_mxfp8_bf16": ([_MXP, _MXP, I64, I64, I64, P, I64, P, I64, P, P], ctypes.c_int),
    "o_proj_mxfp8": ([_MXP, _MXP, _MXP, I64, I32, I32, I32, I32, P, P, P, P, P, P, I64, P, P], ctypes.c_int),
    "o_proj_mxfp8_noalloc": ([_MXP, _MXP, _MXP, I64, I32, I32, I32, I32, P, P, P], ctypes.c_int),
    "o_proj_mxfp8_from_bf16": ([P, I64, _MXP, _MXP, I64, I32, I32, I32, I32, P, P, P, P, P, P, I64, P, P],
                               ctypes.c_int),
}

# capacity of the library-held z buffer of o_proj_mxfp8_noalloc (include/mxq.h)
NOALLOC_Z_BYTES = 2 << 20
NOALLOC_SF_BYTES = 64 << 10


def load():
    """Load libmxq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmxq is not built ({LIB_PATH} missing); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmxq takes device tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != 0:
        detail = load().mxq_last_error_string().decode() if status == 5 else ""
        raise MxqError(status, where, detail)


def abi_version() -> int:
    return int(load().mxq_abi_version())


def workspace_bytes() -> int:
    """Bytes of the split workspace of the large-T GEMMs on the current device."""
    return int(load().mxq_workspace_bytes())


_workspaces = {}


def workspace_for(stream=None) -> Optional[torch.Tensor]:
    """The zero-filled split workspace this module keeps for one CUDA stream, created on its
    first use. Calls ordered on one stream may share it (the library leaves its flags zero);
    concurrent streams each get their own. Under stream capture a workspace is not created (the
    capture would own its memory): there it is None unless a call on the same stream made it
    before the capture began."""
    s = torch.cuda.current_stream() if stream is None else stream
    key = (s.device.index if hasattr(s, "device") else torch.cuda.current_device(), _stream(s).value)
    ws = _workspaces.get(key)
    if ws is None:
        if torch.cuda.is_current_stream_capturing():
            return None
        ws = torch.zeros(workspace_bytes(), dtype=torch.uint8, device=s.device if hasattr(s, "device") else "cuda")
        _workspaces[key] = ws
    return ws


def _ws(workspace, stream):
    """(pointer, bytes) for a workspace argument: None = this stream's own, False = none."""
    if workspace is None:
        workspace = workspace_for(stream)
    if workspace is None or workspace is False:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def sf_bytes(layout: int, M: int, K: int) -> int:
    return int(load().mxq_sf_bytes(layout, M, K))


def status_bytes() -> int:
    return int(load().mxq_status_bytes())


def empty_sf(layout: int, M: int, K: int, device="cuda") -> torch.Tensor:
    n = sf_bytes(layout, M, K)
    if n == 0:
        raise ValueError(f"no scale layout {layout} for [{M}, {K}]")
    return torch.empty(n, dtype=torch.uint8, device=device)


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(status_bytes() // 4, dtype=torch.int32, device=device)


def check_status(status: Optional[torch.Tensor], stream=None) -> None:
    _check(load().mxq_check_status(_ptr(status), _stream(stream)), "mxq_check_status")


@dataclass
class MXFP8:
    """An MXFP8 operand: E4M3 bytes [rows, cols] (uint8) and UE8M0 scales in `layout`."""
    data: torch.Tensor
    sf: torch.Tensor
    layout: int = SF_TILED_128X4

    def c(self) -> MxTensorC:
        d = self.data
        assert d.dtype == torch.uint8 and d.dim() == 2 and d.stride(1) == 1
        return MxTensorC(d.data_ptr(), self.sf.data_ptr(), self.layout, d.shape[0], d.shape[1], d.stride(0))


# ---- the five operations -----------------------------------------------------------------
def mxfp8_quantize(x: torch.Tensor, q: torch.Tensor, sf_rowmajor=None, sf_packed=None, sf_128x4=None,
                   stream=None) -> None:
    """x bf16 [M, K] -> q uint8 [M, K] + any subset of the three scale layouts."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert q.dtype == torch.uint8 and q.dim() == 2 and q.stride(1) == 1
    M, K = x.shape
    _check(load().mxfp8_quantize(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(sf_rowmajor),
                                 _ptr(sf_packed), _ptr(sf_128x4), _stream(stream)), "mxfp8_quantize")


def quantize(x: torch.Tensor, layouts=(SF_TILED_128X4,), stream=None):
    """Allocate outputs and quantize. Returns (q, {layout: sf})."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sfs = {lay: empty_sf(lay, M, K, x.device) for lay in layouts}
    mxfp8_quantize(x, q, sfs.get(SF_ROWMAJOR_U8), sfs.get(SF_PACKED_I32_MN), sfs.get(SF_TILED_128X4), stream)
    return q, sfs


def rmsnorm_dual_out(x: torch.Tensor, gamma: torch.Tensor, eps: float, y: torch.Tensor, yq: torch.Tensor,
                     sf_packed=None, sf_rowmajor=None, sf_128x4=None, stream=None) -> None:
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    T, H = x.shape
    assert y.shape == (T, H) and y.is_contiguous() and yq.shape == (T, H) and yq.is_contiguous()
    _check(load().rmsnorm_dual_out(_ptr(x), _ptr(gamma), float(eps), T, H, x.stride(0), _ptr(y), _ptr(yq),
                                   _ptr(sf_packed), _ptr(sf_rowmajor), _ptr(sf_128x4), _stream(stream)),
           "rmsnorm_dual_out")


def wo_a_einsum_mxfp8(o: MXFP8, wa: MXFP8, T: int, G: int, Na: int, Ka: int, z_q=None, z_sf_128x4=None,
                      z_sf_packed=None, z_bf16=None, status=None, stream=None, workspace=None) -> None:
    """workspace: None = the stream's own split workspace, False = none, or a tensor."""
    oc, wc = o.c(), wa.c()
    wp, wn = _ws(workspace, stream)
    _check(load().wo_a_einsum_mxfp8(ctypes.byref(oc), ctypes.byref(wc), T, G, Na, Ka, _ptr(z_q), _ptr(z_sf_128x4),
                                    _ptr(z_sf_packed), _ptr(z_bf16), wp, wn, _ptr(status), _stream(stream)),
           "wo_a_einsum_mxfp8")


def gemm_mxfp8_bf16(a: MXFP8, b: MXFP8, out: torch.Tensor, status=None, stream=None, workspace=None) -> None:
    M, K = a.data.shape
    N = b.data.shape[0]
    assert out.dtype == torch.bfloat16 and out.stride(1) == 1
    ac, bc = a.c(), b.c()
    wp, wn = _ws(workspace, stream)
    _check(load().gemm_mxfp8_bf16(ctypes.byref(ac), ctypes.byref(bc), M, N, K, _ptr(out), out.stride(0), wp, wn,
                                  _ptr(status), _stream(stream)), "gemm_mxfp8_bf16")


def o_proj_mxfp8(o: MXFP8, wa: MXFP8, wb: MXFP8, T: int, G: int, Na: int, Ka: int, Nb: int, z_q, z_sf_128x4,
                 out: torch.Tensor, z_sf_packed=None, z_bf16=None, status=None, stream=None, workspace=None) -> None:
    oc, ac, bc = o.c(), wa.c(), wb.c()
    wp, wn = _ws(workspace, stream)
    _check(load().o_proj_mxfp8(ctypes.byref(oc), ctypes.byref(ac), ctypes.byref(bc), T, G, Na, Ka, Nb, _ptr(z_q),
                               _ptr(z_sf_128x4), _ptr(z_sf_packed), _ptr(z_bf16), _ptr(out), wp, wn, _ptr(status),
                               _stream(stream)), "o_proj_mxfp8")


def o_proj_mxfp8_noalloc(o: MXFP8, wa: MXFP8, wb: MXFP8, T: int, G: int, Na: int, Ka: int, Nb: int,
                         out: torch.Tensor, status=None, stream=None) -> None:
    """o_proj_mxfp8 with z held in the library's fixed buffer (no z arguments, nothing allocated)."""
    oc, ac, bc = o.c(), wa.c(), wb.c()
    _check(load().o_proj_mxfp8_noalloc(ctypes.byref(oc), ctypes.byref(ac), ctypes.byref(bc), T, G, Na, Ka, Nb,
                                       _ptr(out), _ptr(status), _stream(stream)), "o_proj_mxfp8_noalloc")


def o_proj_mxfp8_from_bf16(o: torch.Tensor, wa: MXFP8, wb: MXFP8, T: int, G: int, Na: int, Ka: int, Nb: int, z_q,
                           z_sf_128x4, out: torch.Tensor, z_sf_packed=None, z_bf16=None, status=None,
                           stream=None, workspace=None) -> None:
    """The _o_proj pair from bf16 o: wo_a quantizes o in the kernel (no quantize launch).
    workspace: None = the stream's own split workspace, False = none, or a tensor."""
    assert o.dtype == torch.bfloat16 and o.dim() == 2 and o.stride(1) == 1
    ac, bc = wa.c(), wb.c()
    wp, wn = _ws(workspace, stream)
    _check(load().o_proj_mxfp8_from_bf16(_ptr(o), o.stride(0), ctypes.byref(ac), ctypes.byref(bc), T, G, Na, Ka, Nb,
                                         _ptr(z_q), _ptr(z_sf_128x4), _ptr(z_sf_packed), _ptr(z_bf16), _ptr(out),
                                         wp, wn, _ptr(status), _stream(stream)), "o_proj_mxfp8_from_bf16")


def selftest_wait_timeout(limit_us: int, status: torch.Tensor, stream=None) -> None:
    """Launch the bounded-wait self-test: a wait that runs out after limit_us and reports a timeout."""
    _check(load().mxq_selftest_wait_timeout(limit_us, _ptr(status), _stream(stream)), "mxq_selftest_wait_timeout")


def selftest_hold_sms(sm_pairs: int, hold_us: int, stream=None) -> None:
    """Occupy `sm_pairs` SM pairs for hold_us microseconds (a clock-bounded diagnostic kernel)."""
    _check(load().mxq_selftest_hold_sms(sm_pairs, hold_us, _stream(stream)), "mxq_selftest_hold_sms")
