"""Oracle for the MXFP8 activation chain -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline / ``--impl
reference`` legs may import this package. The product library never calls it, and it never
calls the product library: the two share no code, header, table or constant.

The arithmetic lives in ``mxq_oracle.cpp`` (plain fp64 C++, compiled here with g++); this
module only builds that file and marshals numpy arrays through ctypes. The one piece of
method logic written in Python is :func:`o_proj_chain`, which calls the C++ steps in the
order the pages give for ``_o_proj``: wo_a einsum -> bf16 z -> MXFP8 z -> wo_b GEMM.

Sources: vLLM pages "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input" (Overview,
Claims, Validation, Details) and "[Perf][DSv4.1] Keep activations MXFP8 between DeepGEMM
kernels" (Purpose: diagrams, per-layer table, Pieces).

Pinning status (each pin is a ``-m "not gpu"`` test in ``tests/test_oracle_pins.py``):
  e4m3_decode / e4m3_encode / ue8m0_from_amax / quantize_bf16 / bf16_round / gemm_nt /
  einsum_wo_a / rmsnorm / sf_to_128x4: pinned.
  sf_pack_i32 (int32-packed MN-major byte order and padding): parity unpinned beyond its own
  definition (pack/unpack identity); no external consumer of that layout exists here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxq_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with g++ (OpenMP when available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if not (force or stale):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        sigs = {
            "orc_abi_version": ([], ctypes.c_int),
            "orc_num_threads": ([], ctypes.c_int),
            "orc_set_num_threads": ([ctypes.c_int], None),
            "orc_bf16_to_f64": ([P, I, P], None),
            "orc_f64_to_bf16": ([P, I, P], None),
            "orc_e4m3_decode": ([P, I, P], None),
            "orc_e4m3_encode": ([P, I, P], None),
            "orc_ue8m0_from_amax": ([P, I, P], None),
            "orc_quantize_bf16": ([P, I, I, I, P, P], None),
            "orc_sf_pack_i32": ([P, I, I, P], None),
            "orc_sf_unpack_i32": ([P, I, I, P], None),
            "orc_sf_128x4_bytes": ([I, I], ctypes.c_int64),
            "orc_sf_to_128x4": ([P, I, I, P], None),
            "orc_sf_from_128x4": ([P, I, I, P], None),
            "orc_dequant": ([P, P, I, I, P], None),
            "orc_gemm_nt": ([P, P, I, I, I, P], None),
            "orc_einsum_wo_a": ([P, P, I, I, I, I, P], None),
            "orc_rmsnorm": ([P, P, ctypes.c_double, I, I, I, P], None),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


# ---- element-wise formats -------------------------------------------------------------------
def bf16_to_f64(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    out = np.empty(x.shape, np.float64)
    _load().orc_bf16_to_f64(_p(x), x.size, _p(out))
    return out


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns, round to nearest even, one rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_f64_to_bf16(_p(x), x.size, _p(out))
    return out


def e4m3_decode(c: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_e4m3_decode(_p(c), c.size, _p(out))
    return out


def e4m3_encode(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64)
    out = np.empty(q.shape, np.uint8)
    _load().orc_e4m3_encode(_p(q), q.size, _p(out))
    return out


def ue8m0_from_amax(amax: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(amax, dtype=np.float64)
    out = np.empty(a.shape, np.uint8)
    _load().orc_ue8m0_from_amax(_p(a), a.size, _p(out))
    return out


# ---- quantizer and layouts ----------------------------------------------------------------
def quantize_bf16(x: np.ndarray):
    """x: uint16 bf16 bits [M, K] -> (q uint8 [M, K], sf uint8 [M, K/32] row-major)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    M, K = x.shape
    assert K % 32 == 0
    q = np.empty((M, K), np.uint8)
    sf = np.empty((M, K // 32), np.uint8)
    _load().orc_quantize_bf16(_p(x), M, K, K, _p(q), _p(sf))
    return q, sf


def sf_pack_i32(sf: np.ndarray) -> np.ndarray:
    """row-major [M, Kg] -> int32-packed MN-major words [Kg/4, ceil(M/4)*4] (uint32)."""
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    M, Kg = sf.shape
    assert Kg % 4 == 0
    out = np.empty((Kg // 4, -(-M // 4) * 4), np.uint32)
    _load().orc_sf_pack_i32(_p(sf), M, Kg, _p(out))
    return out


def sf_unpack_i32(packed: np.ndarray, M: int, Kg: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint32)
    out = np.empty((M, Kg), np.uint8)
    _load().orc_sf_unpack_i32(_p(packed), M, Kg, _p(out))
    return out


def sf_128x4_bytes(M: int, Kg: int) -> int:
    return int(_load().orc_sf_128x4_bytes(M, Kg))


def sf_to_128x4(sf: np.ndarray) -> np.ndarray:
    """row-major [M, Kg] -> flat uint8 F8_128x4 buffer of ceil(M/128)*128 * ceil(Kg/4)*4 bytes."""
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    M, Kg = sf.shape
    out = np.empty(sf_128x4_bytes(M, Kg), np.uint8)
    _load().orc_sf_to_128x4(_p(sf), M, Kg, _p(out))
    return out


def sf_from_128x4(buf: np.ndarray, M: int, Kg: int) -> np.ndarray:
    buf = np.ascontiguousarray(buf, dtype=np.uint8).reshape(-1)
    assert buf.size >= sf_128x4_bytes(M, Kg)
    out = np.empty((M, Kg), np.uint8)
    _load().orc_sf_from_128x4(_p(buf), M, Kg, _p(out))
    return out


# ---- contractions ---------------------------------------------------------------------------
def dequant(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    M, K = q.shape
    assert sf.shape == (M, K // 32)
    out = np.empty((M, K), np.float64)
    _load().orc_dequant(_p(q), _p(sf), M, K, _p(out))
    return out


def gemm_nt(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    C = np.empty((M, N), np.float64)
    _load().orc_gemm_nt(_p(A), _p(B), M, N, K, _p(C))
    return C


def einsum_wo_a(o: np.ndarray, wa: np.ndarray, G: int) -> np.ndarray:
    o = np.ascontiguousarray(o, dtype=np.float64)
    wa = np.ascontiguousarray(wa, dtype=np.float64)
    T, GK = o.shape
    GN, Ka = wa.shape
    assert GK == G * Ka and GN % G == 0
    Na = GN // G
    z = np.empty((T, G * Na), np.float64)
    _load().orc_einsum_wo_a(_p(o), _p(wa), T, G, Na, Ka, _p(z))
    return z


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    gamma = np.ascontiguousarray(gamma, dtype=np.uint16)
    T, H = x.shape
    assert gamma.shape == (H,)
    y = np.empty((T, H), np.float64)
    _load().orc_rmsnorm(_p(x), _p(gamma), float(eps), T, H, H, _p(y))
    return y


def o_proj_chain(o_q, o_sf, wa_q, wa_sf, wb_q, wb_sf, G: int):
    """The `_o_proj` pair as the pages state it, in fp64.

    z_ref = einsum(deq(o), deq(wa)); z_bf16 = RNE_bf16(z_ref); (zq, zsf) = quantize(z_bf16);
    out_ref = deq(zq) . deq(wb)^T.  Inputs are MXFP8 bytes with row-major scales; the rows of
    o may be any subset of the token rows (each row is independent).
    Returns dict(z_ref, z_bf16, zq, zsf, out_ref).
    """
    o_d = dequant(o_q, o_sf)
    wa_d = dequant(wa_q, wa_sf)
    z_ref = einsum_wo_a(o_d, wa_d, G)
    del o_d
    z_bf16 = bf16_round(z_ref)
    zq, zsf = quantize_bf16(z_bf16)
    wb_d = dequant(wb_q, wb_sf)
    out_ref = gemm_nt(dequant(zq, zsf), wb_d)
    return {"z_ref": z_ref, "z_bf16": z_bf16, "zq": zq, "zsf": zsf, "out_ref": out_ref}
