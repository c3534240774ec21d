"""o_proj_mxfp8_noalloc (z in the library's fixed buffer) against o_proj_mxfp8 (z in caller
tensors): the same kernels on the same inputs, so the outputs must agree bit for bit. Two calls
in a row reuse the buffer; the second must not see anything of the first."""
import pytest
import torch

from mxfp8_activation_quant_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    from mxfp8_activation_quant_gb300 import build

    build.build()
    import mxfp8_activation_quant_gb300 as m

    assert torch.cuda.is_available(), "GPU tests need CUDA"
    m.load()
    return m


def _setup(mxq, dev):
    def mx(x):
        q, s = mxq.quantize(x, layouts=(mxq.SF_TILED_128X4,))
        return mxq.MXFP8(q, s[mxq.SF_TILED_128X4])
    return mx, mx(synth.wo_a_weight(5, device=dev)), mx(synth.wo_b_weight(5, device=dev))


def _reference(mxq, O, WA, WB, T, dev):
    zq = torch.empty((T, synth.KB), dtype=torch.uint8, device=dev)
    zsf = mxq.empty_sf(mxq.SF_TILED_128X4, T, synth.KB, dev)
    out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device=dev)
    mxq.o_proj_mxfp8(O, WA, WB, T, synth.G, synth.NA, synth.KA, synth.NB, zq, zsf, out)
    return out


def test_noalloc_matches_o_proj_on_two_calls_in_a_row(mxq):
    dev = torch.device("cuda", 0)
    mx, WA, WB = _setup(mxq, dev)
    status = mxq.new_status(dev)
    results = []
    for seed, T in [(11, 256), (12, 7)]:  # the buffer's largest case, then a small one
        O = mx(synth.o_proj_activation(seed, T, device=dev))
        out = torch.full((T, synth.NB), float("nan"), dtype=torch.bfloat16, device=dev)
        mxq.o_proj_mxfp8_noalloc(O, WA, WB, T, synth.G, synth.NA, synth.KA, synth.NB, out, status=status)
        results.append((O, T, out))
    torch.cuda.synchronize()
    mxq.check_status(status)
    for O, T, out in results:
        want = _reference(mxq, O, WA, WB, T, dev)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), f"T={T}"


def test_noalloc_small_z_width_above_384_tokens(mxq):
    """With a narrow z (G * Na = 1024) the buffer admits up to 2048 tokens, so the pair runs on
    the large-T CTA-pair kernel; without a split workspace that kernel takes whole tiles, and the
    bytes equal o_proj_mxfp8's without a workspace."""
    dev = torch.device("cuda", 0)
    T, G, Na, Ka, Nb = 1000, 1, 1024, 512, 256

    def mx(x):
        q, s = mxq.quantize(x, layouts=(mxq.SF_TILED_128X4,))
        return mxq.MXFP8(q, s[mxq.SF_TILED_128X4])

    WA = mx(synth.normal_bf16(21, 3, G * Na, Ka, Ka ** -0.5, device=dev))
    WB = mx(synth.normal_bf16(21, 4, Nb, G * Na, (G * Na) ** -0.5, device=dev))
    O = mx(synth.normal_bf16(21, 1, T, G * Ka, 1.0, device=dev))
    out = torch.full((T, Nb), float("nan"), dtype=torch.bfloat16, device=dev)
    mxq.o_proj_mxfp8_noalloc(O, WA, WB, T, G, Na, Ka, Nb, out)
    zq = torch.empty((T, G * Na), dtype=torch.uint8, device=dev)
    zsf = mxq.empty_sf(mxq.SF_TILED_128X4, T, G * Na, dev)
    want = torch.empty_like(out)
    mxq.o_proj_mxfp8(O, WA, WB, T, G, Na, Ka, Nb, zq, zsf, want, workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))


def test_noalloc_call_allocates_nothing(mxq):
    """A warm call changes neither torch's allocation count nor the device's free memory."""
    dev = torch.device("cuda", 0)
    mx, WA, WB = _setup(mxq, dev)
    T = 16
    O = mx(synth.o_proj_activation(14, T, device=dev))
    out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device=dev)
    mxq.o_proj_mxfp8_noalloc(O, WA, WB, T, synth.G, synth.NA, synth.KA, synth.NB, out)  # warm
    torch.cuda.synchronize()
    allocs = torch.cuda.memory_stats(dev).get("allocation.all.allocated", 0)
    free = torch.cuda.mem_get_info(dev)[0]
    for _ in range(3):
        mxq.o_proj_mxfp8_noalloc(O, WA, WB, T, synth.G, synth.NA, synth.KA, synth.NB, out)
    torch.cuda.synchronize()
    assert torch.cuda.memory_stats(dev).get("allocation.all.allocated", 0) == allocs
    assert torch.cuda.mem_get_info(dev)[0] == free


def test_noalloc_refuses_shapes_beyond_its_buffer(mxq):
    dev = torch.device("cuda", 0)
    mx, WA, WB = _setup(mxq, dev)
    T = 257
    O = mx(synth.o_proj_activation(13, T, device=dev))
    out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device=dev)
    with pytest.raises(mxq.MxqError) as e:
        mxq.o_proj_mxfp8_noalloc(O, WA, WB, T, synth.G, synth.NA, synth.KA, synth.NB, out)
    assert e.value.status == 2
