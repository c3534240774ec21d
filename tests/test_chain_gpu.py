"""The second producer -> consumer pair of the pages ("[Perf][DSv4.1] Keep activations MXFP8
between DeepGEMM kernels", Purpose, before/after diagrams): RMSNorm emits y as bf16 and as
MXFP8, and the MXFP8 GEMM `fused_wqa_wkv` consumes the MXFP8 y directly. The GEMM width is not
on the pages; 2048 output features stand in for it (synth.WQKV_N).

  * y_q and its F8_128x4 scales equal the standalone quantizer applied to the kernel's own bf16 y;
  * the GEMM output is within 1e-2 relative Frobenius of the fp64 oracle chain
    (RMSNorm -> RNE bf16 -> MXFP8 -> dequantized GEMM)."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, bits_to_f64, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    from mxfp8_activation_quant_gb300 import build

    build.build()
    import mxfp8_activation_quant_gb300 as m

    assert torch.cuda.is_available(), "GPU tests need CUDA"
    m.load()
    return m


@pytest.mark.parametrize("T", [1, 64, 300, 1024])
def test_rmsnorm_feeds_mxfp8_gemm(mxq, oracle, T):
    from mxfp8_activation_quant_gb300 import synth

    H, N = synth.RMS_H, synth.WQKV_N
    x = synth.rmsnorm_input(7, T, device="cuda")
    g = synth.rmsnorm_gamma(7, device="cuda")
    w = synth.wqa_wkv_weight(7, device="cuda")
    wq, wsf = mxq.quantize(w, layouts=(mxq.SF_TILED_128X4,))
    W = mxq.MXFP8(wq, wsf[mxq.SF_TILED_128X4])
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    yq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    ysf = mxq.empty_sf(mxq.SF_TILED_128X4, T, H)
    mxq.rmsnorm_dual_out(x, g, synth.RMS_EPS, y, yq, sf_128x4=ysf)
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    mxq.gemm_mxfp8_bf16(mxq.MXFP8(yq, ysf), W, out)
    torch.cuda.synchronize()
    # the MXFP8 y is exactly the quantizer's output on the kernel's own bf16 y
    q2, s2 = mxq.quantize(y, layouts=(mxq.SF_TILED_128X4,))
    torch.cuda.synchronize()
    assert torch.equal(q2, yq) and torch.equal(s2[mxq.SF_TILED_128X4], ysf)
    # the whole chain against the oracle's own
    y_ref = oracle.bf16_round(oracle.rmsnorm(bf16_bits(x), bf16_bits(g), synth.RMS_EPS))
    yq_o, ysf_o = oracle.quantize_bf16(y_ref)
    wq_o, wsf_o = oracle.quantize_bf16(bf16_bits(w))
    assert np.array_equal(wq.cpu().numpy(), wq_o)
    out_ref = oracle.gemm_nt(oracle.dequant(yq_o, ysf_o), oracle.dequant(wq_o, wsf_o))
    assert rel_fro(bits_to_f64(bf16_bits(out)), out_ref) <= 1e-2
