"""The algorithmic bytes and FLOPs behind bench.py's roofline fractions, pinned to figures worked
out by hand from the shapes of the DeepSeek-V4.1 `_o_proj` pair ("[Perf][DSv4.1] MegaAttn: wo_a
writes wo_b's MXFP8 input", the decode and prefill sweeps) and of the standalone quantizer and
the RMSNorm dual-output producer ("[Perf][DSv4.1] Keep activations MXFP8 between DeepGEMM
kernels"): every figure below is a product of the shapes written out by hand, not another call
of the function under test."""
import bench


def test_o_proj_flops_per_token():
    # wo_a: 8 groups x 1024 features x 4096 inputs; wo_b: 5120 x 8192; 2 FLOP per multiply-add
    assert bench.wo_a_flops(1) + bench.wo_b_flops(1) == 150_994_944
    assert bench.wo_a_flops(4096) == 274_877_906_944
    assert bench.wo_b_flops(4096) == 343_597_383_680


def test_o_proj_bytes():
    # weights once, E4M3 plus one UE8M0 byte per 32 elements: 34,603,008 + 43,253,760
    assert bench.wo_a_bytes(0) + bench.wo_b_bytes(0) == 77_856_768
    # per token: o 32768 + 1024 scale bytes read, z 8192 + 256 written by wo_a and read by wo_b,
    # out 10240 bytes of bf16 written
    per_token = 32768 + 1024 + 2 * (8192 + 256) + 10240
    assert (bench.wo_a_bytes(1) + bench.wo_b_bytes(1)) - 77_856_768 == per_token == 60_928


def test_quantizer_bytes():
    # [32768, 8192] bf16 in, E4M3 out, one scale layout: 3 + 1/32 bytes per element
    assert bench.quant_bytes(32768, 8192) == 813_694_976
    assert bench.quant_bytes(4096, 8192) == 101_711_872
    # each further scale layout adds one byte per 32 elements
    assert bench.quant_bytes(4096, 8192, layouts=3) - bench.quant_bytes(4096, 8192) == 2 * 4096 * 256


def test_rmsnorm_bytes():
    # [8192, 5120]: x read, y bf16 written, y E4M3 written, one packed scale byte per 32, gamma once
    assert bench.rms_bytes(8192) == 8192 * 5120 * 5 + 8192 * 160 + 10240 == 211_036_160
    assert bench.rms_bytes(1024) == 1024 * 5120 * 5 + 1024 * 160 + 10240
