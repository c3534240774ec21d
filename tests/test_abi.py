"""The C-ABI library loads, exports every symbol include/mxq.h declares, and rejects bad
arguments on the host (these calls return before any CUDA work, so no GPU is needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxq.h")


@pytest.fixture(scope="module")
def lib():
    from mxfp8_activation_quant_gb300 import _lib, build

    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"MXQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(lib):
    from mxfp8_activation_quant_gb300 import _lib

    names = declared_functions()
    assert len(names) == 16, names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES)


def test_version_and_status_strings(lib):
    assert lib.mxq_abi_version() == 3
    for code, name in [(0, b"MXQ_OK"), (2, b"MXQ_ERR_UNSUPPORTED_SHAPE"), (6, b"MXQ_ERR_TIMEOUT")]:
        assert lib.mxq_status_string(code) == name
    assert lib.mxq_status_bytes() >= 4
    # four 128 KB partial slots, 128 bytes of flags and 128 bytes of tickets per SM pair
    assert lib.mxq_workspace_bytes() > 0 and lib.mxq_workspace_bytes() % (4 * 128 * 1024 + 256) == 0


def test_sf_bytes_match_oracle_layout_sizes(lib, oracle):
    for M, K in [(1, 8192), (129, 8192), (300, 160), (8193, 5120)]:
        assert lib.mxq_sf_bytes(0, M, K) == M * (K // 32)
        assert lib.mxq_sf_bytes(2, M, K) == oracle.sf_128x4_bytes(M, K // 32)
        if K % 128 == 0:
            assert lib.mxq_sf_bytes(1, M, K) == (K // 128) * (-(-M // 4) * 4) * 4
        else:
            assert lib.mxq_sf_bytes(1, M, K) == 0
    assert lib.mxq_sf_bytes(0, 4, 48) == 0 and lib.mxq_sf_bytes(9, 4, 64) == 0


FAKE = 0x7F0000000000  # never dereferenced: every call below fails validation first


def test_quantize_argument_errors(lib):
    q = lib.mxfp8_quantize
    assert q(None, 4, 64, 64, FAKE, 64, FAKE, None, None, None) == 1            # null input
    assert q(FAKE, 4, 64, 64, FAKE, 64, None, None, None, None) == 1            # no scale output
    assert q(FAKE, 0, 64, 64, FAKE, 64, FAKE, None, None, None) == 1            # M = 0
    assert q(FAKE, 4, 48, 48, FAKE, 48, FAKE, None, None, None) == 2            # K % 32
    assert q(FAKE, 4, 96, 96, FAKE, 96, None, FAKE, None, None) == 2            # packed, K % 128
    assert q(FAKE, 4, 64, 32, FAKE, 64, FAKE, None, None, None) == 2            # ldx < K
    assert q(FAKE + 2, 4, 64, 64, FAKE, 64, FAKE, None, None, None) == 3        # misaligned x
    assert q(FAKE, 4, 64, 68, FAKE, 64, FAKE, None, None, None) == 3            # ldx*2 % 16
    assert q(FAKE, 4, 64, 64, FAKE, 64, FAKE + 8, None, None, None) == 3        # misaligned sf


def test_rmsnorm_argument_errors(lib):
    r = lib.rmsnorm_dual_out
    assert r(FAKE, FAKE, 1e-6, 4, 5120, 5120, FAKE, FAKE, None, None, None, None) == 1
    assert r(FAKE, FAKE, 1e-6, 4, 5000, 5000, FAKE, FAKE, FAKE, None, None, None) == 2
    assert r(FAKE, FAKE, 1e-6, 4, 32768, 32768, FAKE, FAKE, FAKE, None, None, None) == 2
    assert r(FAKE, FAKE, -1.0, 4, 5120, 5120, FAKE, FAKE, FAKE, None, None, None) == 1
    assert r(FAKE, FAKE + 4, 1e-6, 4, 5120, 5120, FAKE, FAKE, FAKE, None, None, None) == 3


def test_gemm_argument_errors(lib):
    from mxfp8_activation_quant_gb300._lib import MxTensorC

    def mx(rows, cols, layout=2, data=FAKE, ld=None):
        return MxTensorC(data, FAKE, layout, rows, cols, ld if ld is not None else cols)

    o, wa, wb = mx(8, 32768), mx(8192, 4096), mx(5120, 8192)
    B = ctypes.byref
    e = lib.wo_a_einsum_mxfp8
    W0 = (None, 0)  # no split workspace
    assert e(B(o), B(wa), 8, 8, 1024, 4096, FAKE, None, None, None, *W0, None, None) == 1    # z_q w/o scales
    assert e(B(o), B(wa), 8, 8, 1024, 4096, None, None, None, None, *W0, None, None) == 1    # no output
    assert e(B(mx(8, 32768, layout=0)), B(wa), 8, 8, 1024, 4096, FAKE, FAKE, None, None, *W0, None, None) == 4
    assert e(B(o), B(wa), 8, 8, 1000, 4096, FAKE, FAKE, None, None, *W0, None, None) == 2    # Na % 128
    assert e(B(o), B(wa), 9, 8, 1024, 4096, FAKE, FAKE, None, None, *W0, None, None) == 2    # rows != T
    assert e(B(mx(8, 32768, data=FAKE + 1)), B(wa), 8, 8, 1024, 4096, FAKE, FAKE, None, None, *W0, None, None) == 3
    assert e(B(o), B(wa), 8, 8, 1024, 4096, FAKE, FAKE, None, None, FAKE, 16, None, None) == 1  # workspace too small
    assert e(B(o), B(wa), 8, 8, 1024, 4096, FAKE, FAKE, None, None, FAKE + 8, 1 << 30, None, None) == 3
    g = lib.gemm_mxfp8_bf16
    assert g(B(mx(8, 8192)), B(wb), 8, 5120, 8192, None, 5120, *W0, None, None) == 1
    assert g(B(mx(8, 8192)), B(mx(5000, 8192)), 8, 5000, 8192, FAKE, 5000, *W0, None, None) == 2
    assert g(B(mx(8, 8192)), B(wb), 8, 5120, 8192, FAKE, 5124, *W0, None, None) == 3          # ldo*2 % 16
    assert g(B(mx(8, 8192)), B(wb), 8, 5120, 8192, FAKE, 5120, FAKE, 16, None, None) == 1     # workspace too small
    p = lib.o_proj_mxfp8
    assert p(B(o), B(wa), B(wb), 8, 8, 1024, 4096, 5120, None, FAKE, None, None, FAKE, *W0, None, None) == 1
    assert p(B(o), B(wa), B(mx(5120, 8192, layout=1)), 8, 8, 1024, 4096, 5120, FAKE, FAKE, None, None, FAKE,
             *W0, None, None) == 4
    assert p(B(o), B(wa), B(wb), 8, 8, 1024, 4096, 5120, FAKE, FAKE, None, None, FAKE, FAKE + 4, 1 << 30, None,
             None) == 3                                                                      # misaligned workspace


def test_o_proj_noalloc_argument_errors(lib):
    from mxfp8_activation_quant_gb300._lib import NOALLOC_Z_BYTES, MxTensorC

    def mx(rows, cols):
        return MxTensorC(FAKE, FAKE, 2, rows, cols, cols)

    B = ctypes.byref
    n = lib.o_proj_mxfp8_noalloc
    t_max = NOALLOC_Z_BYTES // 8192  # 256 tokens for G * Na = 8192
    # shapes beyond the fixed buffer are refused before any CUDA call
    for T in (t_max + 1, 4096):
        assert n(B(mx(T, 32768)), B(mx(8192, 4096)), B(mx(5120, 8192)), T, 8, 1024, 4096, 5120, FAKE, None,
                 None) == 2
    assert n(B(mx(0, 32768)), B(mx(8192, 4096)), B(mx(5120, 8192)), 0, 8, 1024, 4096, 5120, FAKE, None, None) == 1
    assert n(B(mx(4, 32768)), B(mx(8192, 4096)), B(mx(5120, 8192)), 4, 8, 1000, 4096, 5120, FAKE, None, None) == 2


def test_o_proj_from_bf16_argument_errors(lib):
    from mxfp8_activation_quant_gb300._lib import MxTensorC

    def mx(rows, cols):
        return MxTensorC(FAKE, FAKE, 2, rows, cols, cols)

    B = ctypes.byref
    f = lib.o_proj_mxfp8_from_bf16
    args = (B(mx(8192, 4096)), B(mx(5120, 8192)))
    ws = (None, 0)
    assert f(FAKE, 32768, *args, 4, 8, 1000, 4096, 5120, FAKE, FAKE, None, None, FAKE, *ws, None, None) == 2  # Na
    assert f(None, 32768, *args, 4, 8, 1024, 4096, 5120, FAKE, FAKE, None, None, FAKE, *ws, None, None) == 1
    assert f(FAKE, 32000, *args, 4, 8, 1024, 4096, 5120, FAKE, FAKE, None, None, FAKE, *ws, None, None) == 2  # ld_o
    assert f(FAKE + 2, 32768, *args, 4, 8, 1024, 4096, 5120, FAKE, FAKE, None, None, FAKE, *ws, None, None) == 3
    assert f(FAKE, 32772, *args, 4, 8, 1024, 4096, 5120, FAKE, FAKE, None, None, FAKE, *ws, None, None) == 3  # ld_o*2 % 16
    assert f(FAKE, 32768, *args, 4, 8, 1024, 4096, 5120, FAKE, FAKE, None, None, FAKE, FAKE, 16, None, None) == 1  # ws size


def test_selftest_argument_errors(lib):
    assert lib.mxq_selftest_wait_timeout(1000, None, None) == 1
    assert lib.mxq_selftest_wait_timeout(0, FAKE, None) == 1
    assert lib.mxq_selftest_wait_timeout(2000000, FAKE, None) == 1  # the limit stays within 1 s
    assert lib.mxq_selftest_wait_timeout(1000, FAKE + 4, None) == 3


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every call raises; nothing falls back to another implementation."""
    from mxfp8_activation_quant_gb300 import _lib

    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libmxq.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.abi_version()
    with pytest.raises(RuntimeError, match="not built"):
        _lib.workspace_bytes()


def test_host_tensors_are_refused(lib):
    """The binding passes device pointers only: a host tensor is an error, not a CPU path."""
    import torch

    from mxfp8_activation_quant_gb300 import _lib

    x = torch.zeros(4, 32, dtype=torch.bfloat16)
    q = torch.zeros(4, 32, dtype=torch.uint8)
    with pytest.raises(ValueError, match="device tensors"):
        _lib.mxfp8_quantize(x, q)
