"""RMSNorm dual-output producer on the GPU (page "[Perf][DSv4.1] Keep activations MXFP8
between DeepGEMM kernels", Purpose: mega_mhc's RMSNorm emitting bf16 y and (y_fp8, y_gemm_sf)).

bf16 y within one bf16 ulp of the fp64 oracle; the MXFP8 y bit-identical to the standalone
quantizer applied to the GPU's own bf16 y, and to the oracle's quantizer wherever the GPU's y
equals the oracle's correctly rounded y."""
import numpy as np
import pytest
import torch

from helpers import Guarded, bf16_bits, bf16_ulp, bits_to_f64, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    from mxfp8_activation_quant_gb300 import build

    build.build()
    import mxfp8_activation_quant_gb300 as m

    assert torch.cuda.is_available(), "GPU tests need CUDA"
    m.load()
    return m


@pytest.mark.parametrize("T", [1, 7, 64, 129, 1024, 8192])
def test_rmsnorm_dual_out(mxq, oracle, T):
    from mxfp8_activation_quant_gb300 import synth

    check_rmsnorm(mxq, oracle, T, synth.RMS_H)


# The block shape follows the row count (256 threads a row up to 512 rows, 160 up to 2048,
# 128 beyond): each shape at widths that leave idle threads, partial scale words and the
# largest accepted width.
@pytest.mark.parametrize("T,H", [(5, 16384), (3, 96), (600, 2080), (1500, 16384), (2600, 96), (2600, 7168)])
def test_rmsnorm_dual_out_widths(mxq, oracle, T, H):
    check_rmsnorm(mxq, oracle, T, H)


def check_rmsnorm(mxq, oracle, T, H):
    from mxfp8_activation_quant_gb300 import synth

    eps = synth.RMS_EPS
    x = synth.rmsnorm_input(0, T, H)
    gamma = synth.rmsnorm_gamma(0, H)
    y = Guarded(T * H * 2)
    yq = Guarded(T * H)
    packed = H % 128 == 0  # the int32-packed layout needs whole 4-group words
    pk = Guarded(mxq.sf_bytes(1, T, H)) if packed else None
    rm = Guarded(mxq.sf_bytes(0, T, H))
    tl = Guarded(mxq.sf_bytes(2, T, H))
    mxq.rmsnorm_dual_out(x.cuda(), gamma.cuda(), eps, y.view(torch.bfloat16, (T, H)), yq.view(shape=(T, H)),
                         pk.body if packed else None, rm.body, tl.body)
    torch.cuda.synchronize()
    for g in (y, yq, pk, rm, tl):
        assert g is None or g.intact()

    # (1) bf16 y within one bf16 ulp of the fp64 reference
    y_ref = oracle.rmsnorm(bf16_bits(x), bf16_bits(gamma), eps)
    y_gpu_bits = u8(y.body).view(np.uint16).reshape(T, H)
    y_gpu = bits_to_f64(y_gpu_bits)
    err = np.abs(y_gpu - y_ref) / bf16_ulp(y_ref)
    assert err.max() <= 1.0, f"max error {err.max()} ulp"

    # (2) MXFP8 y == standalone quantizer on the GPU's own bf16 y (both layouts)
    yg = y.view(torch.bfloat16, (T, H))
    q2 = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    rm2 = mxq.empty_sf(0, T, H)
    pk2 = mxq.empty_sf(1, T, H) if packed else None
    tl2 = mxq.empty_sf(2, T, H)
    mxq.mxfp8_quantize(yg, q2, rm2, pk2, tl2)
    torch.cuda.synchronize()
    assert torch.equal(q2, yq.view(shape=(T, H)))
    assert torch.equal(rm2, rm.body) and torch.equal(tl2, tl.body)
    assert not packed or torch.equal(pk2, pk.body)

    # (3) against the oracle's quantizer on the oracle's own RNE(y_ref), in every 32-element
    # group where the two y agree (quantization is local to a group)
    y_rne = oracle.bf16_round(y_ref)
    same = np.all((y_rne == y_gpu_bits).reshape(T, H // 32, 32), axis=2)
    assert same.mean() > 0.9
    oq, osf = oracle.quantize_bf16(y_rne)
    assert np.array_equal(u8(yq.body).reshape(T, H // 32, 32)[same], oq.reshape(T, H // 32, 32)[same])
    assert np.array_equal(u8(rm.body).reshape(T, H // 32)[same], osf[same])


def test_rmsnorm_constant_rows(mxq):
    """x = c everywhere, gamma = 1: y = c / sqrt(c^2 + eps) (closed form)."""
    T, H = 4, 5120
    x = torch.full((T, H), 3.0, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    yq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    mxq.rmsnorm_dual_out(x, g, 1e-6, y, yq, sf_packed=mxq.empty_sf(1, T, H))
    torch.cuda.synchronize()
    want = torch.tensor(3.0 / np.sqrt(9.0 + 1e-6), dtype=torch.float32).to(torch.bfloat16)
    assert torch.all(y == want.cuda())
