"""Failure detection without a GPU fault: a bounded wait on a barrier that nothing arrives on runs
out, the kernel records MXQ_ERR_TIMEOUT in the status word, mxq_check_status reports it, and the
context keeps working afterwards (the same bounded-wait routine guards every pipeline wait)."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    from mxfp8_activation_quant_gb300 import build

    build.build()
    import mxfp8_activation_quant_gb300 as m

    assert torch.cuda.is_available(), "GPU tests need CUDA"
    m.load()
    return m


def test_wait_runs_out_and_is_reported(mxq):
    st = mxq.new_status()
    t0 = time.perf_counter()
    mxq.selftest_wait_timeout(5000, st)  # 5 ms
    with pytest.raises(mxq.MxqError) as e:
        mxq.check_status(st)  # synchronizes
    assert e.value.status == 6  # MXQ_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.005
    # the first recorded error stays until the caller clears the word
    mxq.selftest_wait_timeout(1000, st)
    with pytest.raises(mxq.MxqError):
        mxq.check_status(st)
    st.zero_()
    mxq.check_status(st)


def test_context_still_works_after_a_timeout(mxq):
    from mxfp8_activation_quant_gb300 import synth

    x = synth.quantizer_input(3, 64, 1024, device="cuda")
    before = mxq.quantize(x, layouts=(mxq.SF_TILED_128X4,))
    torch.cuda.synchronize()
    st = mxq.new_status()
    mxq.selftest_wait_timeout(1000, st)
    with pytest.raises(mxq.MxqError):
        mxq.check_status(st)
    after = mxq.quantize(x, layouts=(mxq.SF_TILED_128X4,))
    torch.cuda.synchronize()
    assert torch.equal(before[0], after[0])
    assert torch.equal(before[1][mxq.SF_TILED_128X4], after[1][mxq.SF_TILED_128X4])
