"""Failure detection on the GPU without a fault: a pipeline wait that nobody
completes runs out (the same bounded mbarrier wait every kernel uses), the
device status word reports NVFP4_ERR_DEVICE_TIMEOUT, and the context keeps
working."""
import pytest
import torch

import oracle
import synthdata
from parity import check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    import nvfp4_block_scaled_act_gb300 as m
    m.load_library()
    return m


def test_pipeline_wait_timeout_is_reported_and_the_context_survives(nv):
    assert nv.nvfp4_device_status() == 0
    nv.nvfp4_selftest_wait_timeout()
    assert nv.nvfp4_device_status() == 6  # NVFP4_ERR_DEVICE_TIMEOUT, and cleared by the read
    assert nv.nvfp4_device_status() == 0
    # the next call on the same context runs and is correct
    case = synthdata.decode_case(4, 256, 512, seed=7)
    w = case.w_parts[0]
    W = nv.quantize_weight(w.to("cuda"))
    out = nv.nvfp4_linear_w4a16(case.x[:4].to("cuda"), W.codes, W.scales, nv.nvfp4_make_alpha(None, W.g), 256, 512)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status() == 0
    g = oracle.global_scale(w)
    wc, ws = oracle.quantize(w, g)
    check_close(out.cpu(), oracle.linear_w4a16(case.x[:4], wc, ws, 256, 512, oracle.alpha_w4a16(g)), "after timeout")
