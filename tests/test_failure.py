"""GPU: the failure path of the kernels' bounded waits.  A self-test block waits on a barrier that
nothing arrives on; the wait runs out after about a second, reports it through the per-device
error word (swa_check_device raises SWA_ERR_DEVICE_TIMEOUT), and the context stays usable: the
word is cleared by the read and the next attention call runs and matches the oracle."""
import numpy as np
import pytest
import torch

import swa_inputs as si
from oracle import swa_oracle as orc
from test_parity import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives(swa):
    lib = swa.load()
    dev = torch.device("cuda:0")
    swa.swa_check_device()  # start from a clear word
    assert lib.swa_selftest_wait_timeout(torch.cuda.current_stream(dev).cuda_stream) == 0
    with pytest.raises(swa.SwaError) as ei:
        swa.swa_check_device()
    assert ei.value.code == 5  # SWA_ERR_DEVICE_TIMEOUT
    swa.swa_check_device()  # the read cleared the word
    case = si.tiny_case()
    inputs = si.make_inputs(case)
    gpu = run_gpu(swa, case, inputs)
    ref = orc.oracle_backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"], case.W,
                              case.softmax_scale)
    check_against_oracle(case, gpu, ref)
    assert np.isfinite(gpu["o"]).all()
