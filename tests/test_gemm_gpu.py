"""The _o_proj GEMMs on the GPU (page "[Perf][DSv4.1] MegaAttn: wo_a writes wo_b's MXFP8 input",
Overview / Validation / Details).

  * exact small cases: integer-valued E4M3 operands make every dot product exact in fp32, so
    the bf16 output must equal the rounded exact result bit for bit (catches any operand,
    scale-layout or descriptor error);
  * wo_a bf16 z within 4e-3 relative Frobenius of the fp64 oracle; the fused MXFP8 z bytes and
    scales identical to the standalone quantizer applied to the same call's bf16 z (the pages'
    claim that wo_b gets the very same FP8 bytes and scales as before the fusion);
  * the whole _o_proj output within 1e-2 relative Frobenius of the oracle's own chain.
Token counts follow the pages' tests: 1, 129, 8193 tokens and M in {1, 4, 7, 64, 300}, plus the
decode and prefill sweeps."""
import ctypes
import re
import time

import numpy as np
import pytest
import torch

from helpers import Guarded, bf16_bits, bits_to_f64, rel_fro, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    from mxfp8_activation_quant_gb300 import build

    build.build()
    import mxfp8_activation_quant_gb300 as m

    assert torch.cuda.is_available(), "GPU tests need CUDA"
    m.load()
    return m


def gpu_mx(mxq, x_bf16):
    q, sfs = mxq.quantize(x_bf16.cuda(), layouts=(mxq.SF_TILED_128X4,))
    return mxq.MXFP8(q, sfs[mxq.SF_TILED_128X4])


def int_matrix(rng, rows, cols, lo=-4, hi=4):
    return torch.from_numpy(rng.integers(lo, hi + 1, (rows, cols)).astype(np.float32)).to(torch.bfloat16)


# ------------------------------------------------------------------------------------------
# exact small GEMMs (both orientations, split and unsplit K, ragged token tails)
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T,N,K", [(1, 128, 128), (1, 256, 1152), (2, 128, 640), (7, 128, 256), (16, 256, 512), (32, 128, 1024), (64, 128, 1024),
                                   (96, 128, 1024), (100, 128, 256), (128, 256, 2048), (200, 256, 1024),
                                   (250, 128, 1024), (256, 128, 512), (300, 256, 256), (384, 128, 384),
                                   (513, 256, 512),
                                   # more than 384 tokens with N % 256 != 0: the one-CTA
                                   # normal-orientation kernel (128 tokens x 128 features per tile)
                                   (513, 384, 512), (1000, 640, 1024), (8193, 128, 256),
                                   # wo_b's shape at three token bands, and 65 k-blocks (no power of
                                   # two divides them: K stays unsplit)
                                   (33, 5120, 8192), (100, 5120, 8192), (64, 5120, 8320)])
def test_gemm_exact_integers(mxq, oracle, T, N, K):
    rng = np.random.default_rng(T * 7 + N + K)
    a = int_matrix(rng, T, K)
    b = int_matrix(rng, N, K)
    A, B = gpu_mx(mxq, a), gpu_mx(mxq, b)
    out = Guarded(T * N * 2)
    mxq.gemm_mxfp8_bf16(A, B, out.view(torch.bfloat16, (T, N)))
    torch.cuda.synchronize()
    assert out.intact()
    exact = a.double().numpy() @ b.double().numpy().T
    want = oracle.bf16_round(exact)
    got = u8(out.body).view(np.uint16).reshape(T, N)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} of {T * N} differ; first {bad[:4].tolist()}: " \
                          f"got {bits_to_f64(got[tuple(bad[0])])} want {exact[tuple(bad[0])]}"


# ------------------------------------------------------------------------------------------
# stream-K split of the CTA-pair GEMM (T > 384 with a workspace)
# ------------------------------------------------------------------------------------------
SK_SLOTS_PER_PAIR = 4 * 128 * 1024  # partial sums: two segments x two CTAs, 128 x 256 fp32
SK_PER_PAIR = SK_SLOTS_PER_PAIR + 256  # + 128 bytes of ready flags and 128 of tickets


def _flags_zero(mxq, ws):
    """The flag and ticket bytes (after the partial slots of every SM pair) are all zero."""
    pairs = ws.numel() // SK_PER_PAIR
    return bool((ws[pairs * SK_SLOTS_PER_PAIR:] == 0).all())


def _slots_written(ws):
    pairs = ws.numel() // SK_PER_PAIR
    return bool((ws[: pairs * SK_SLOTS_PER_PAIR] != 0).any())


@pytest.mark.parametrize("T,N,K", [(1000, 5120, 8192), (2000, 5120, 8192)])
def test_split_k_exact_integers(mxq, oracle, T, N, K):
    """The split tail (80 and 160 tiles of 256 x 256 on the SM pairs, 64 k-blocks each: the last
    wave and the remainder are cut into equal k-block ranges, and the pair that starts a tile adds
    the partial sums of the others): with integer operands every partial sum is exact, so the
    output equals the exact product bit for bit and the whole-tile (no workspace) result, and the
    flags end at zero. T = 1000 also leaves the last tile's second CTA without tokens."""
    rng = np.random.default_rng(T + N + K)
    a = int_matrix(rng, T, K)
    b = int_matrix(rng, N, K)
    A, B = gpu_mx(mxq, a), gpu_mx(mxq, b)
    ws = torch.zeros(mxq.workspace_bytes(), dtype=torch.uint8, device="cuda")
    out = Guarded(T * N * 2)
    mxq.gemm_mxfp8_bf16(A, B, out.view(torch.bfloat16, (T, N)), workspace=ws)
    whole = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    mxq.gemm_mxfp8_bf16(A, B, whole, workspace=False)
    torch.cuda.synchronize()
    assert out.intact() and _flags_zero(mxq, ws)
    assert _slots_written(ws)  # partial slots were written: the split ran
    got = u8(out.body).view(np.uint16).reshape(T, N)
    want = oracle.bf16_round(a.double().numpy() @ b.double().numpy().T)
    assert np.array_equal(got, want)
    assert np.array_equal(got, bf16_bits(whole))


def test_split_k_completes_while_other_work_holds_sms(mxq, oracle):
    """No pair of the split tail waits for one that has not started: with all but 16 SM pairs held
    by another stream's kernel for 1.5 s (longer than the pipelines' 1 s bounded waits), the split
    GEMM (76 pairs at T = 2000) still completes while that kernel holds its SMs, with MXQ_OK, the
    exact product and the flags and tickets back at zero."""
    T, N, K = 2000, 5120, 8192
    rng = np.random.default_rng(29)
    a = int_matrix(rng, T, K)
    b = int_matrix(rng, N, K)
    A, B = gpu_mx(mxq, a), gpu_mx(mxq, b)
    ws = torch.zeros(mxq.workspace_bytes(), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    st = mxq.new_status()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s_hold, s_gemm = torch.cuda.Stream(), torch.cuda.Stream()
    e_hold, e_gemm = torch.cuda.Event(), torch.cuda.Event()
    torch.cuda.synchronize()
    mxq.selftest_hold_sms(sms // 2 - 16, 1_500_000, stream=s_hold)
    e_hold.record(s_hold)
    time.sleep(0.05)  # the holding kernel takes its SMs first
    mxq.gemm_mxfp8_bf16(A, B, out, status=st, stream=s_gemm, workspace=ws)
    e_gemm.record(s_gemm)
    e_gemm.synchronize()
    held_still = not e_hold.query()
    torch.cuda.synchronize()
    mxq.check_status(st)
    assert held_still, "the GEMM did not run beside the holding kernel"
    assert _flags_zero(mxq, ws) and _slots_written(ws)
    want = oracle.bf16_round(a.double().numpy() @ b.double().numpy().T)
    assert np.array_equal(bf16_bits(out), want)


def test_split_k_grouped_fused_epilogue(mxq, oracle):
    """The split tail under the fused z epilogue: a grouped einsum (G = 2, 2560 features, 8192
    deep, T = 1000: 80 tiles) with integer operands gives bf16 z equal to the rounded exact
    result, MXFP8 z equal to the standalone quantizer applied to that z, and the same bytes as
    whole tiles."""
    T, G, Na, Ka = 1000, 2, 2560, 8192
    rng = np.random.default_rng(5)
    o = int_matrix(rng, T, G * Ka, -3, 3)
    wa = int_matrix(rng, G * Na, Ka, -3, 3)
    O, WA = gpu_mx(mxq, o), gpu_mx(mxq, wa)
    ws = torch.zeros(mxq.workspace_bytes(), dtype=torch.uint8, device="cuda")
    outs = []
    for w in (ws, False):
        zq = Guarded(T * G * Na)
        ztl = Guarded(mxq.sf_bytes(2, T, G * Na))
        zb = Guarded(T * G * Na * 2)
        mxq.wo_a_einsum_mxfp8(O, WA, T, G, Na, Ka, zq.view(shape=(T, G * Na)), ztl.body, None,
                              zb.view(torch.bfloat16, (T, G * Na)), workspace=w)
        outs.append((zq, ztl, zb))
    torch.cuda.synchronize()
    assert _flags_zero(mxq, ws)
    assert _slots_written(ws)  # the split ran
    (zq, ztl, zb), (zq_w, ztl_w, zb_w) = outs
    for gbuf in (zq, ztl, zb, zq_w, ztl_w, zb_w):
        assert gbuf.intact()
    a, b = o.double().numpy(), wa.double().numpy()
    exact = np.concatenate([a[:, g * Ka:(g + 1) * Ka] @ b[g * Na:(g + 1) * Na].T for g in range(G)], axis=1)
    got = u8(zb.body).view(np.uint16).reshape(T, G * Na)
    assert np.array_equal(got, oracle.bf16_round(exact))
    q2, sfs = mxq.quantize(zb.view(torch.bfloat16, (T, G * Na)), layouts=(2,))
    torch.cuda.synchronize()
    assert torch.equal(q2, zq.view(shape=(T, G * Na))) and torch.equal(sfs[2], ztl.body)
    assert torch.equal(zq.body, zq_w.body) and torch.equal(ztl.body, ztl_w.body) and torch.equal(zb.body, zb_w.body)


def test_o_proj_workspace_serves_wo_b_only(mxq):
    """At a shape where wo_a alone takes the split tail (G = 2, 2560 features, 8192 deep, T = 1000:
    80 tiles of 64 k-blocks) and so does wo_b (80 tiles of 40 k-blocks), o_proj_mxfp8 gives the
    workspace to wo_b only: wo_b, a programmatic dependent, takes its tickets while wo_a may still
    run, so the two must not share flags. The call equals wo_a_einsum_mxfp8 without a workspace
    followed by gemm_mxfp8_bf16 with it, byte for byte, and the flags end at zero."""
    T, G, Na, Ka, Nb = 1000, 2, 2560, 8192, 5120
    rng = np.random.default_rng(41)
    O = gpu_mx(mxq, int_matrix(rng, T, G * Ka, -3, 3))
    WA = gpu_mx(mxq, int_matrix(rng, G * Na, Ka, -3, 3))
    WB = gpu_mx(mxq, int_matrix(rng, Nb, G * Na, -2, 2))
    ws = torch.zeros(mxq.workspace_bytes(), dtype=torch.uint8, device="cuda")

    def bufs():
        return (torch.empty((T, G * Na), dtype=torch.uint8, device="cuda"), mxq.empty_sf(2, T, G * Na),
                torch.empty((T, Nb), dtype=torch.bfloat16, device="cuda"))

    st = mxq.new_status()
    a = bufs()
    for _ in range(3):  # repeated calls reuse the flags and tickets
        mxq.o_proj_mxfp8(O, WA, WB, T, G, Na, Ka, Nb, a[0], a[1], a[2], status=st, workspace=ws)
    b = bufs()
    mxq.wo_a_einsum_mxfp8(O, WA, T, G, Na, Ka, z_q=b[0], z_sf_128x4=b[1], status=st, workspace=False)
    mxq.gemm_mxfp8_bf16(mxq.MXFP8(b[0], b[1]), WB, b[2], status=st, workspace=ws)
    torch.cuda.synchronize()
    mxq.check_status(st)
    assert _flags_zero(mxq, ws) and _slots_written(ws)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_split_k_o_proj_deterministic(mxq, weights):
    """The pair at T = 1000 (wo_b split, wo_a in whole tiles) repeats its bytes exactly, stays
    within one bf16 rounding of the whole-tile result, and leaves the flags zero."""
    from mxfp8_activation_quant_gb300 import synth

    T = 1000
    O = gpu_mx(mxq, synth.o_proj_activation(3, T))
    ws = torch.zeros(mxq.workspace_bytes(), dtype=torch.uint8, device="cuda")
    res = []
    for w in (ws, ws, False):
        zq = torch.empty((T, synth.KB), dtype=torch.uint8, device="cuda")
        ztl = mxq.empty_sf(mxq.SF_TILED_128X4, T, synth.KB, "cuda")
        out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device="cuda")
        mxq.o_proj_mxfp8(O, weights.WA, weights.WB, T, synth.G, synth.NA, synth.KA, synth.NB, zq, ztl, out,
                         workspace=w)
        res.append((zq, ztl, out))
    torch.cuda.synchronize()
    assert _flags_zero(mxq, ws)
    (zq1, ztl1, out1), (zq2, ztl2, out2), (_, _, out3) = res
    assert torch.equal(zq1, zq2) and torch.equal(ztl1, ztl2) and torch.equal(out1, out2)
    # only the fp32 summation order differs: a bf16 rounding step here and there
    a, b = out1.float(), out3.float()
    assert float((a - b).abs().max()) <= 2.0 ** -7 * float(b.abs().max())
    assert float((a - b).norm()) <= 2e-3 * float(b.norm())


@pytest.mark.parametrize("T", [5, 130, 260])
def test_gemm_random_scales(mxq, oracle, T):
    from mxfp8_activation_quant_gb300 import synth

    N, K = 256, 1024
    a = synth.quantizer_input(11, T, K=K)
    b = synth.normal_bf16(12, 1, N, K, 0.05)
    A, B = gpu_mx(mxq, a), gpu_mx(mxq, b)
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    mxq.gemm_mxfp8_bf16(A, B, out)
    torch.cuda.synchronize()
    aq, asf = oracle.quantize_bf16(bf16_bits(a))
    bq, bsf = oracle.quantize_bf16(bf16_bits(b))
    ref = oracle.gemm_nt(oracle.dequant(aq, asf), oracle.dequant(bq, bsf))
    got = bits_to_f64(bf16_bits(out))
    # fp32 accumulation + one bf16 rounding: half a bf16 ulp of each output plus fp32 sum error
    scale = oracle.gemm_nt(np.abs(oracle.dequant(aq, asf)), np.abs(oracle.dequant(bq, bsf)))
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + scale * K * 2.0 ** -23 + 1e-30)


# ------------------------------------------------------------------------------------------
# small grouped einsum: fused MXFP8 epilogue == standalone quantizer on the same bf16 z
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1, 2, 5, 129, 260])
def test_wo_a_small_groups(mxq, oracle, T):
    from mxfp8_activation_quant_gb300 import synth

    G, Na, Ka = 2, 256, 512
    o = synth.quantizer_input(21, T, K=G * Ka)
    wa = synth.normal_bf16(22, 1, G * Na, Ka, 1.0 / np.sqrt(Ka))
    O, WA = gpu_mx(mxq, o), gpu_mx(mxq, wa)
    zq = Guarded(T * G * Na)
    ztl = Guarded(mxq.sf_bytes(2, T, G * Na))
    zpk = Guarded(mxq.sf_bytes(1, T, G * Na))
    zb = Guarded(T * G * Na * 2)
    mxq.wo_a_einsum_mxfp8(O, WA, T, G, Na, Ka, zq.view(shape=(T, G * Na)), ztl.body, zpk.body,
                          zb.view(torch.bfloat16, (T, G * Na)))
    torch.cuda.synchronize()
    for g in (zq, ztl, zpk, zb):
        assert g.intact()
    oq, osf = oracle.quantize_bf16(bf16_bits(o))
    wq, wsf = oracle.quantize_bf16(bf16_bits(wa))
    z_ref = oracle.einsum_wo_a(oracle.dequant(oq, osf), oracle.dequant(wq, wsf), G)
    z_gpu = bits_to_f64(u8(zb.body).view(np.uint16).reshape(T, G * Na))
    assert rel_fro(z_gpu, z_ref) <= 4e-3
    # fused quantization == standalone quantizer applied to this call's bf16 z
    q2, sfs = mxq.quantize(zb.view(torch.bfloat16, (T, G * Na)), layouts=(1, 2))
    torch.cuda.synchronize()
    assert torch.equal(q2, zq.view(shape=(T, G * Na)))
    assert torch.equal(sfs[2], ztl.body) and torch.equal(sfs[1], zpk.body)


def test_wo_a_grouped_normal_orientation(mxq, oracle):
    """A grouped einsum whose feature count per group is not a multiple of 256 (G = 2, Na = 384)
    with more than 384 tokens runs on the one-CTA normal-orientation kernel. Integer operands make
    every sum exact: the bf16 z equals the rounded exact product bit for bit, and the fused MXFP8
    z and both its scale layouts equal the standalone quantizer applied to that z."""
    T, G, Na, Ka = 700, 2, 384, 512
    rng = np.random.default_rng(17)
    o = int_matrix(rng, T, G * Ka, -3, 3)
    wa = int_matrix(rng, G * Na, Ka, -3, 3)
    O, WA = gpu_mx(mxq, o), gpu_mx(mxq, wa)
    zq = Guarded(T * G * Na)
    ztl = Guarded(mxq.sf_bytes(2, T, G * Na))
    zpk = Guarded(mxq.sf_bytes(1, T, G * Na))
    zb = Guarded(T * G * Na * 2)
    mxq.wo_a_einsum_mxfp8(O, WA, T, G, Na, Ka, zq.view(shape=(T, G * Na)), ztl.body, zpk.body,
                          zb.view(torch.bfloat16, (T, G * Na)))
    torch.cuda.synchronize()
    for gbuf in (zq, ztl, zpk, zb):
        assert gbuf.intact()
    a, b = o.double().numpy(), wa.double().numpy()
    exact = np.concatenate([a[:, g * Ka:(g + 1) * Ka] @ b[g * Na:(g + 1) * Na].T for g in range(G)], axis=1)
    got = u8(zb.body).view(np.uint16).reshape(T, G * Na)
    assert np.array_equal(got, oracle.bf16_round(exact))
    q2, sfs = mxq.quantize(zb.view(torch.bfloat16, (T, G * Na)), layouts=(1, 2))
    torch.cuda.synchronize()
    assert torch.equal(q2, zq.view(shape=(T, G * Na)))
    assert torch.equal(sfs[2], ztl.body) and torch.equal(sfs[1], zpk.body)
    # and the oracle's quantizer on the oracle's own rounded product gives the same bytes
    oq, osf = oracle.quantize_bf16(oracle.bf16_round(exact))
    assert np.array_equal(u8(zq.body).reshape(T, G * Na), oq)
    assert np.array_equal(oracle.sf_from_128x4(u8(ztl.body), T, G * Na // 32), osf)


def launched_kernels(fn):
    """Names of the device kernels `fn` launches (torch.profiler / CUPTI); None when the
    profiler records no kernels at all in this environment."""
    from torch.profiler import ProfilerActivity, profile

    for _ in range(2):  # a process's first profiling session may come back empty
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if "cuda" in str(getattr(e, "device_type", "")).lower()]
        if names:
            return names
    return None


@pytest.mark.parametrize("T", [100, 128])
def test_uneven_split_kernel_runs_at_wo_b_shape(mxq, oracle, T):
    """wo_b's shape in the 64 < T <= 128 band takes the swap-AB kernel with K cut over three
    cluster ranks (the power-of-two split would leave SMs idle); check that this instantiation is
    the one that ran, and that its integer-operand output is exact."""
    N, K = 5120, 8192
    rng = np.random.default_rng(T + 3)
    a = int_matrix(rng, T, K)
    b = int_matrix(rng, N, K)
    A, B = gpu_mx(mxq, a), gpu_mx(mxq, b)
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    names = launched_kernels(lambda: mxq.gemm_mxfp8_bf16(A, B, out))
    if names is None:
        pytest.skip("the profiler records no device kernels here")
    gemm = [n for n in names if "gemm_mxf8" in n]
    assert len(gemm) == 1, names
    assert re.search(r"gemm_mxf8_kernel<128, 6, (true|1), 0, 3>", gemm[0]), gemm[0]
    want = oracle.bf16_round(a.double().numpy() @ b.double().numpy().T)
    assert np.array_equal(bf16_bits(out), want)


# ------------------------------------------------------------------------------------------
# full DeepSeek-V4.1 _o_proj shapes
# ------------------------------------------------------------------------------------------
class Weights:
    pass


@pytest.fixture(scope="module")
def weights(mxq, oracle):
    from mxfp8_activation_quant_gb300 import synth

    w = Weights()
    wa = synth.wo_a_weight(0, device="cuda")
    wb = synth.wo_b_weight(0, device="cuda")
    w.WA, w.WB = gpu_mx(mxq, wa), gpu_mx(mxq, wb)
    waq, wasf = oracle.quantize_bf16(bf16_bits(wa))
    wbq, wbsf = oracle.quantize_bf16(bf16_bits(wb))
    w.wa_d = oracle.dequant(waq, wasf)
    w.wb_d = oracle.dequant(wbq, wbsf)
    # the GPU quantized the same bf16 weights the oracle did (bit-exact quantizer)
    assert np.array_equal(u8(w.WA.data), waq) and np.array_equal(u8(w.WB.data), wbq)
    return w


def oracle_chain(oracle, w, o_bits):
    from mxfp8_activation_quant_gb300 import synth

    oq, osf = oracle.quantize_bf16(o_bits)
    z_ref = oracle.einsum_wo_a(oracle.dequant(oq, osf), w.wa_d, synth.G)
    zq, zsf = oracle.quantize_bf16(oracle.bf16_round(z_ref))
    out_ref = oracle.gemm_nt(oracle.dequant(zq, zsf), w.wb_d)
    return z_ref, out_ref


def run_o_proj(mxq, w, O, T, with_bf16=True):
    from mxfp8_activation_quant_gb300 import synth

    Kb = synth.KB
    zq = torch.empty((T, Kb), dtype=torch.uint8, device="cuda")
    ztl = mxq.empty_sf(2, T, Kb)
    zb = torch.empty((T, Kb), dtype=torch.bfloat16, device="cuda") if with_bf16 else None
    out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device="cuda")
    mxq.o_proj_mxfp8(O, w.WA, w.WB, T, synth.G, synth.NA, synth.KA, synth.NB, zq, ztl, out, z_bf16=zb)
    torch.cuda.synchronize()
    return zq, ztl, zb, out


@pytest.mark.parametrize("T", [1, 2, 4, 7, 8, 16, 24, 33, 64, 100, 128, 129, 256, 300, 384])
def test_o_proj_decode_shapes(mxq, oracle, weights, T):
    from mxfp8_activation_quant_gb300 import synth

    o = synth.o_proj_activation(0, T)
    O = gpu_mx(mxq, o)
    zq, ztl, zb, out = run_o_proj(mxq, weights, O, T)
    z_ref, out_ref = oracle_chain(oracle, weights, bf16_bits(o))
    assert rel_fro(bits_to_f64(bf16_bits(zb)), z_ref) <= 4e-3
    assert rel_fro(bits_to_f64(bf16_bits(out)), out_ref) <= 1e-2
    q2, sfs = mxq.quantize(zb, layouts=(2,))
    torch.cuda.synchronize()
    assert torch.equal(q2, zq) and torch.equal(sfs[2], ztl)
    # the MXFP8-only call (no bf16 z written) gives the same bytes and output
    zq2, ztl2, _, out2 = run_o_proj(mxq, weights, O, T, with_bf16=False)
    assert torch.equal(zq2, zq) and torch.equal(ztl2, ztl) and torch.equal(out2, out)


@pytest.mark.parametrize("T", [385, 512, 1000, 4096, 8193, 32768])
def test_o_proj_prefill_sampled_rows(mxq, oracle, weights, T):
    """Full-size prefill: the oracle checks the first and last 128-row tiles and 256 seeded
    rows; the fused-vs-standalone identity is checked on every row."""
    from mxfp8_activation_quant_gb300 import synth

    o = synth.o_proj_activation(0, T, device="cuda")
    rows = synth.sample_rows(0, T)
    o_rows = synth.o_proj_activation(0, T, rows=rows)
    assert np.array_equal(bf16_bits(o[rows.cuda()]), bf16_bits(o_rows))
    O = gpu_mx(mxq, o)
    del o
    zq, ztl, zb, out = run_o_proj(mxq, weights, O, T)
    z_ref, out_ref = oracle_chain(oracle, weights, bf16_bits(o_rows))
    r = rows.cuda()
    assert rel_fro(bits_to_f64(bf16_bits(zb[r])), z_ref) <= 4e-3
    assert rel_fro(bits_to_f64(bf16_bits(out[r])), out_ref) <= 1e-2
    q2, sfs = mxq.quantize(zb, layouts=(2,))
    torch.cuda.synchronize()
    assert torch.equal(q2, zq) and torch.equal(sfs[2], ztl)


def test_o_proj_graph_replay(mxq, weights):
    """The two-launch chain captured in a CUDA graph replays to identical bytes."""
    from mxfp8_activation_quant_gb300 import synth

    T = 129
    O = gpu_mx(mxq, synth.o_proj_activation(1, T))
    zq, ztl, _, out = run_o_proj(mxq, weights, O, T, with_bf16=False)
    zq2 = torch.zeros_like(zq)
    ztl2 = torch.zeros_like(ztl)
    out2 = torch.zeros_like(out)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm-up on the capture stream (it also makes its split workspace)
        mxq.o_proj_mxfp8(O, weights.WA, weights.WB, T, synth.G, synth.NA, synth.KA, synth.NB, zq2, ztl2, out2)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mxq.o_proj_mxfp8(O, weights.WA, weights.WB, T, synth.G, synth.NA, synth.KA, synth.NB, zq2, ztl2, out2)
    zq2.zero_()
    ztl2.zero_()
    out2.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(zq2, zq) and torch.equal(ztl2, ztl) and torch.equal(out2, out)


def _kernel_nodes(graph):
    """Kernel nodes of a captured CUDA graph, counted through the driver API."""
    cu = ctypes.CDLL("libcuda.so.1")
    h = ctypes.c_void_p(graph.raw_cuda_graph())
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(h, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert cu.cuGraphGetNodes(h, nodes, ctypes.byref(n)) == 0
    kinds = []
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kinds.append(t.value)
    return sum(k == 0 for k in kinds), len(kinds)  # CU_GRAPH_NODE_TYPE_KERNEL == 0


@pytest.mark.parametrize("T", [1, 256, 4096])
def test_fused_chain_launches_two_kernels(mxq, weights, T):
    """No standalone quantize launch in the fused path: a captured o_proj_mxfp8 holds exactly two
    kernels (wo_a, wo_b), and the unfused chain (wo_a writing bf16 z, the quantizer, wo_b) three."""
    from mxfp8_activation_quant_gb300 import synth

    try:
        g1, g2 = torch.cuda.CUDAGraph(keep_graph=True), torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        pytest.skip("this torch cannot keep the captured graph")
    O = gpu_mx(mxq, synth.o_proj_activation(3, T))
    zq = torch.empty((T, synth.KB), dtype=torch.uint8, device="cuda")
    ztl = mxq.empty_sf(2, T, synth.KB)
    zb = torch.empty((T, synth.KB), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device="cuda")
    Z = mxq.MXFP8(zq, ztl)

    def fused():
        mxq.o_proj_mxfp8(O, weights.WA, weights.WB, T, synth.G, synth.NA, synth.KA, synth.NB, zq, ztl, out)

    def unfused():
        mxq.wo_a_einsum_mxfp8(O, weights.WA, T, synth.G, synth.NA, synth.KA, z_bf16=zb)
        mxq.mxfp8_quantize(zb, zq, None, None, ztl)
        mxq.gemm_mxfp8_bf16(Z, weights.WB, out)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fused()
        unfused()
    torch.cuda.synchronize()
    with torch.cuda.graph(g1):
        fused()
    with torch.cuda.graph(g2):
        unfused()
    assert _kernel_nodes(g1) == (2, 2)
    assert _kernel_nodes(g2) == (3, 3)


@pytest.mark.parametrize("T,pad", [(1, 0), (2, 0), (4, 0), (7, 64), (16, 0), (17, 0), (33, 64), (100, 0), (129, 0),
                                   (256, 0), (300, 64), (384, 0), (385, 0), (1000, 64), (2048, 0), (4096, 0),
                                   (8193, 0)])
def test_o_proj_from_bf16_matches_prequantized(mxq, oracle, weights, T, pad):
    """wo_a quantizing bf16 o in the kernel against mxfp8_quantize(o) followed by o_proj_mxfp8
    (the pages' "pre-quantized == in-kernel"). At every token count both run the same tiles and K
    splits (swap-AB bands up to 384 tokens, the CTA-pair kernel beyond, quantizing in place; at
    2048 tokens its last wave runs in 256 x 128 halves): z,
    both scale layouts, the bf16 z and out are the same bytes. The in-kernel path also meets the
    oracle chain's tolerances (bf16 z within 4e-3, out within 1e-2; sampled rows beyond 384
    tokens). `pad` extra columns make o a strided view."""
    from mxfp8_activation_quant_gb300 import synth

    o_full = torch.zeros((T, synth.G * synth.KA + pad), dtype=torch.bfloat16, device="cuda")
    o = o_full[:, : synth.G * synth.KA]
    o.copy_(synth.o_proj_activation(8, T, device="cuda"))
    st = mxq.new_status()

    def bufs():
        return (torch.empty((T, synth.KB), dtype=torch.uint8, device="cuda"), mxq.empty_sf(2, T, synth.KB),
                mxq.empty_sf(1, T, synth.KB), torch.empty((T, synth.KB), dtype=torch.bfloat16, device="cuda"),
                torch.empty((T, synth.NB), dtype=torch.bfloat16, device="cuda"))

    a = bufs()
    mxq.o_proj_mxfp8_from_bf16(o, weights.WA, weights.WB, T, synth.G, synth.NA, synth.KA, synth.NB, a[0], a[1], a[4],
                               z_sf_packed=a[2], z_bf16=a[3], status=st)
    b = bufs()
    O = gpu_mx(mxq, o.contiguous())
    mxq.o_proj_mxfp8(O, weights.WA, weights.WB, T, synth.G, synth.NA, synth.KA, synth.NB, b[0], b[1], b[4],
                     z_sf_packed=b[2], z_bf16=b[3], status=st)
    torch.cuda.synchronize()
    mxq.check_status(st)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    rows = np.arange(T) if T <= 384 else synth.sample_rows(0, T).numpy()
    o_rows = o.cpu()[torch.from_numpy(rows)]
    z_ref, out_ref = oracle_chain(oracle, weights, bf16_bits(o_rows))
    assert rel_fro(bits_to_f64(bf16_bits(a[3]))[rows], z_ref) <= 4e-3
    assert rel_fro(bits_to_f64(bf16_bits(a[4]))[rows], out_ref) <= 1e-2


@pytest.mark.parametrize("T,G,Na,Ka,Nb", [(600, 2, 512, 1024, 256), (700, 2, 384, 512, 256), (50, 3, 256, 384, 128)])
def test_o_proj_from_bf16_other_shapes(mxq, oracle, T, G, Na, Ka, Nb):
    """The bf16-o pair away from the DeepSeek shapes, with exact integer operands: (600, Na = 512)
    runs the quantizing CTA-pair kernel with every tile in 256 x 128 halves, (700, Na = 384) the
    one-CTA normal-orientation kernel, (50) a swap-AB band with 3 groups. bf16 z equals the
    rounded exact product; the MXFP8 z and its scales equal the standalone quantizer applied to
    that z; and where the tiles are o_proj_mxfp8's (Na a multiple of 256, or T <= 384) every
    output is the bytes of mxfp8_quantize + o_proj_mxfp8."""
    rng = np.random.default_rng(T + G + Na)
    o = int_matrix(rng, T, G * Ka, -3, 3)
    wa = int_matrix(rng, G * Na, Ka, -3, 3)
    wb = int_matrix(rng, Nb, G * Na, -2, 2)
    WA, WB = gpu_mx(mxq, wa), gpu_mx(mxq, wb)
    st = mxq.new_status()

    def bufs():
        return (torch.empty((T, G * Na), dtype=torch.uint8, device="cuda"), mxq.empty_sf(2, T, G * Na),
                torch.empty((T, G * Na), dtype=torch.bfloat16, device="cuda"),
                torch.empty((T, Nb), dtype=torch.bfloat16, device="cuda"))

    a = bufs()
    mxq.o_proj_mxfp8_from_bf16(o.cuda(), WA, WB, T, G, Na, Ka, Nb, a[0], a[1], a[3], z_bf16=a[2], status=st)
    torch.cuda.synchronize()
    mxq.check_status(st)
    od, wad = o.double().numpy(), wa.double().numpy()
    exact = np.concatenate([od[:, g * Ka:(g + 1) * Ka] @ wad[g * Na:(g + 1) * Na].T for g in range(G)], axis=1)
    assert np.array_equal(bf16_bits(a[2]), oracle.bf16_round(exact))
    q2, sfs = mxq.quantize(a[2], layouts=(2,))
    torch.cuda.synchronize()
    assert torch.equal(q2, a[0]) and torch.equal(sfs[2], a[1])
    if Na % 256 == 0 or T <= 384:
        b = bufs()
        mxq.o_proj_mxfp8(gpu_mx(mxq, o), WA, WB, T, G, Na, Ka, Nb, b[0], b[1], b[3], z_bf16=b[2], status=st)
        torch.cuda.synchronize()
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("T,N,K", [(1, 256, 512), (17, 256, 512), (40, 128, 1024), (100, 5120, 8192),
                                   (128, 256, 2048), (300, 256, 1024), (513, 256, 512), (700, 384, 512),
                                   (1000, 5120, 8192)])
def test_gemm_exact_integers_packed_scales(mxq, oracle, T, N, K):
    """The activation's scales as int32-packed MN-major words, at every token band (swap-AB tiles
    of 16 to 128 tokens, the 3-rank split at wo_b's shape, the CTA-pair kernel with and without
    the split tail, the normal orientation): integer operands, so the output equals the exact
    product bit for bit, and equals the output from the F8_128x4 scales."""
    rng = np.random.default_rng(T * 3 + N + K)
    a = int_matrix(rng, T, K)
    b = int_matrix(rng, N, K)
    aq, asf = mxq.quantize(a.cuda(), layouts=(mxq.SF_PACKED_I32_MN, mxq.SF_TILED_128X4))
    A_pk = mxq.MXFP8(aq, asf[mxq.SF_PACKED_I32_MN], mxq.SF_PACKED_I32_MN)
    A_tl = mxq.MXFP8(aq, asf[mxq.SF_TILED_128X4])
    B = gpu_mx(mxq, b)
    ws = torch.zeros(mxq.workspace_bytes(), dtype=torch.uint8, device="cuda")
    out = Guarded(T * N * 2)
    mxq.gemm_mxfp8_bf16(A_pk, B, out.view(torch.bfloat16, (T, N)), workspace=ws)
    ref = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    mxq.gemm_mxfp8_bf16(A_tl, B, ref, workspace=ws)
    torch.cuda.synchronize()
    assert out.intact() and _flags_zero(mxq, ws)
    got = u8(out.body).view(np.uint16).reshape(T, N)
    assert np.array_equal(got, oracle.bf16_round(a.double().numpy() @ b.double().numpy().T))
    assert np.array_equal(got, bf16_bits(ref))


@pytest.mark.parametrize("T", [1, 2, 5, 16, 17, 33, 100, 129, 256, 300, 385, 1000, 4096, 8193])
def test_wo_b_reads_packed_scales(mxq, oracle, weights, T):
    """wo_b taking z with int32-packed MN-major scales (the layout the fused epilogue writes as
    its second output) gives the same bf16 output as with the F8_128x4 scales, standalone and as
    the dependent half of the pair. Against the oracle: the packed words decode (oracle's
    definition of the layout) to the same scales as the tiled ones; the output equals the fp64
    GEMM on this z's bytes and decoded packed scales within one bf16 rounding plus fp32
    summation error; and the chain output is within 1e-2 of the oracle's own chain."""
    from mxfp8_activation_quant_gb300 import synth

    O = gpu_mx(mxq, synth.o_proj_activation(9, T, device="cuda"))
    zq = torch.empty((T, synth.KB), dtype=torch.uint8, device="cuda")
    ztl, zpk = mxq.empty_sf(2, T, synth.KB), mxq.empty_sf(1, T, synth.KB)
    out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device="cuda")
    mxq.o_proj_mxfp8(O, weights.WA, weights.WB, T, synth.G, synth.NA, synth.KA, synth.NB, zq, ztl, out,
                     z_sf_packed=zpk)
    out_pk = torch.empty_like(out)
    mxq.gemm_mxfp8_bf16(mxq.MXFP8(zq, zpk, mxq.SF_PACKED_I32_MN), weights.WB, out_pk)
    out_tl = torch.empty_like(out)
    mxq.gemm_mxfp8_bf16(mxq.MXFP8(zq, ztl), weights.WB, out_tl)
    torch.cuda.synchronize()
    assert torch.equal(out_pk, out_tl)
    # the standalone wo_b (5 stages) splits K like the paired one: same bytes as the pair too
    assert torch.equal(out_pk, out)
    Kg = synth.KB // 32
    sf_pk = oracle.sf_unpack_i32(u8(zpk).view(np.uint32).reshape(Kg // 4, -1), T, Kg)
    assert np.array_equal(sf_pk, oracle.sf_from_128x4(u8(ztl), T, Kg))
    # the oracle on every row up to 384 tokens, on the sampled rows beyond
    rows = np.arange(T) if T <= 384 else synth.sample_rows(0, T).numpy()
    zd = oracle.dequant(u8(zq)[rows], sf_pk[rows])
    ref = oracle.gemm_nt(zd, weights.wb_d)
    scale = oracle.gemm_nt(np.abs(zd), np.abs(weights.wb_d))
    got = bits_to_f64(bf16_bits(out_pk))[rows]
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + scale * synth.KB * 2.0 ** -23 + 1e-30)
    o_rows = synth.o_proj_activation(9, T, rows=torch.from_numpy(rows))
    _, out_ref = oracle_chain(oracle, weights, bf16_bits(o_rows))
    assert rel_fro(got, out_ref) <= 1e-2


def test_status_word_stays_clear(mxq, weights):
    from mxfp8_activation_quant_gb300 import synth

    T = 16
    O = gpu_mx(mxq, synth.o_proj_activation(2, T))
    st = mxq.new_status()
    zq = torch.empty((T, synth.KB), dtype=torch.uint8, device="cuda")
    ztl = mxq.empty_sf(2, T, synth.KB)
    out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device="cuda")
    mxq.o_proj_mxfp8(O, weights.WA, weights.WB, T, synth.G, synth.NA, synth.KA, synth.NB, zq, ztl, out, status=st)
    mxq.check_status(st)
    assert int(st[0]) == 0
