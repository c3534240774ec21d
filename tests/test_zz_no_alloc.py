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


def test_noalloc_refuses_shapes_beyond_its_buffer(mxq):
    dev = torch.device("cuda", 0)
    mx, WA, WB = _setup(mxq, dev)
    T = 257
    O = mx(synth.o_proj_activation(13, T, device=dev))
    out = torch.empty((T, synth.NB), dtype=torch.bfloat16, device=dev)
    with pytest.raises(mxq.MxqError) as e:
        mxq.o_proj_mxfp8_noalloc(O, WA, WB, T, synth.G, synth.NA, synth.KA, synth.NB, out)
    assert e.value.status == 2
