"""Standalone MXFP8 quantizer on the GPU against the oracle: bytes and all three scale
layouts bit-exact (page "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input", Claims:
the standalone mxfp8_quantize launch; scale layouts as stated in include/mxq.h)."""
import numpy as np
import pytest
import torch

from helpers import Guarded, bf16_bits, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    from mxfp8_activation_quant_gb300 import build

    build.build()
    import mxfp8_activation_quant_gb300 as m

    assert torch.cuda.is_available(), "GPU tests need CUDA"
    m.load()
    return m


def run_quantize(mxq, x_dev, ldx=None):
    M, K = x_dev.shape
    q = Guarded(M * K)
    rm = Guarded(mxq.sf_bytes(0, M, K))
    pk = Guarded(mxq.sf_bytes(1, M, K)) if K % 128 == 0 else None
    tl = Guarded(mxq.sf_bytes(2, M, K))
    mxq.mxfp8_quantize(x_dev, q.view(shape=(M, K)), rm.body, pk.body if pk else None, tl.body)
    torch.cuda.synchronize()
    return q, rm, pk, tl


def check_against_oracle(oracle, xbits, q, rm, pk, tl):
    M, K = xbits.shape
    oq, osf = oracle.quantize_bf16(xbits)
    got_q = u8(q.body).reshape(M, K)
    bad = np.argwhere(got_q != oq)
    assert bad.size == 0, f"{len(bad)} E4M3 bytes differ, first at {bad[:5].tolist()}"
    assert np.array_equal(u8(rm.body).reshape(M, K // 32), osf)
    if pk is not None:
        assert np.array_equal(u8(pk.body).view(np.uint32), oracle.sf_pack_i32(osf).reshape(-1))
    assert np.array_equal(u8(tl.body), oracle.sf_to_128x4(osf))
    for g in (q, rm, tl) + ((pk,) if pk is not None else ()):
        assert g.intact(), "write outside the output buffer"


@pytest.mark.parametrize("T", [1, 7, 16, 129, 256, 300, 4096, 8193])
def test_quantize_matches_oracle(mxq, oracle, T):
    from mxfp8_activation_quant_gb300 import synth

    x = synth.quantizer_input(0, T)
    check_against_oracle(oracle, bf16_bits(x), *run_quantize(mxq, x.cuda()))


@pytest.mark.parametrize("K", [32, 96, 160, 1056, 5120])
def test_quantize_ragged_k(mxq, oracle, K):
    from mxfp8_activation_quant_gb300 import synth

    x = synth.quantizer_input(3, 37, K=K)
    check_against_oracle(oracle, bf16_bits(x), *run_quantize(mxq, x.cuda()))


def test_quantize_every_bf16_pattern(mxq, oracle):
    """Each finite bf16 pattern alone in its group (the rest zero), and again inside random
    context groups."""
    b = np.arange(65536, dtype=np.uint32)
    fin = b[((b >> 7) & 0xFF) != 0xFF].astype(np.uint16)
    iso = np.zeros((fin.size, 128), np.uint16)
    iso[:, 5] = fin
    rng = np.random.default_rng(0)
    ctx = rng.choice(fin, size=(fin.size // 32 + 1) * 32 * 4).astype(np.uint16).reshape(-1, 128)
    ctx.reshape(-1)[: fin.size] = fin
    for arr in (iso, ctx):
        x = torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)
        check_against_oracle(oracle, arr, *run_quantize(mxq, x.cuda()))


def test_quantize_strided_input(mxq, oracle):
    from mxfp8_activation_quant_gb300 import synth

    big = synth.quantizer_input(5, 40, K=1024)
    x = big.cuda()[:, 128:640]          # row stride 1024, K = 512
    q, rm, pk, tl = run_quantize(mxq, x)
    check_against_oracle(oracle, bf16_bits(big[:, 128:640]), q, rm, pk, tl)


def test_quantize_full_size_32768(mxq, oracle):
    """T = 32768 x 8192 (the largest quantizer workload): drawn on the GPU by the generator,
    every output compared with the oracle; a row sample is re-drawn on the CPU to show the
    generator gives the oracle the same input on either device."""
    from mxfp8_activation_quant_gb300 import synth

    T = 32768
    x = synth.quantizer_input(0, T, device="cuda")
    rows = synth.sample_rows(0, T, n_random=64)
    assert np.array_equal(bf16_bits(x[rows.cuda()]), bf16_bits(synth.quantizer_input(0, T, rows=rows)))
    q, rm, pk, tl = run_quantize(mxq, x)
    check_against_oracle(oracle, bf16_bits(x), q, rm, pk, tl)


def test_quantize_repeatable(mxq):
    from mxfp8_activation_quant_gb300 import synth

    x = synth.quantizer_input(9, 300).cuda()
    a = run_quantize(mxq, x)
    b = run_quantize(mxq, x)
    for ga, gb in zip(a, b):
        if ga is not None:
            assert torch.equal(ga.body, gb.body)


def test_quantize_graph_replay(mxq):
    """Captured in a CUDA graph and replayed, the call writes the same bytes."""
    from mxfp8_activation_quant_gb300 import synth

    x = synth.quantizer_input(2, 129).cuda()
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    tl = mxq.empty_sf(2, M, K)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mxq.mxfp8_quantize(x, q, None, None, tl)
    torch.cuda.synchronize()
    ref_q, ref_tl = q.clone(), tl.clone()
    q.zero_()
    tl.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mxq.mxfp8_quantize(x, q, None, None, tl)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(q, ref_q) and torch.equal(tl, ref_tl)
