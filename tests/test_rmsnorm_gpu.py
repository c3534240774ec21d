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

    H, eps = synth.RMS_H, synth.RMS_EPS
    x = synth.rmsnorm_input(0, T)
    gamma = synth.rmsnorm_gamma(0)
    y = Guarded(T * H * 2)
    yq = Guarded(T * H)
    pk = Guarded(mxq.sf_bytes(1, T, H))
    rm = Guarded(mxq.sf_bytes(0, T, H))
    tl = Guarded(mxq.sf_bytes(2, T, H))
    mxq.rmsnorm_dual_out(x.cuda(), gamma.cuda(), eps, y.view(torch.bfloat16, (T, H)), yq.view(shape=(T, H)),
                         pk.body, rm.body, tl.body)
    torch.cuda.synchronize()
    for g in (y, yq, pk, rm, tl):
        assert g.intact()

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
    pk2 = mxq.empty_sf(1, T, H)
    tl2 = mxq.empty_sf(2, T, H)
    mxq.mxfp8_quantize(yg, q2, rm2, pk2, tl2)
    torch.cuda.synchronize()
    assert torch.equal(q2, yq.view(shape=(T, H)))
    assert torch.equal(rm2, rm.body) and torch.equal(pk2, pk.body) and torch.equal(tl2, tl.body)

    # (3) against the oracle's quantizer on the oracle's own RNE(y_ref), rows where y agrees
    y_rne = oracle.bf16_round(y_ref)
    same = np.all(y_rne == y_gpu_bits, axis=1)
    assert same.mean() > 0.5
    oq, osf = oracle.quantize_bf16(y_rne[same])
    assert np.array_equal(u8(yq.body).reshape(T, H)[same], oq)
    assert np.array_equal(u8(rm.body).reshape(T, H // 32)[same], osf)


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
