"""Device failure detection on the GPU without a fault: a bounded wait that nothing satisfies
gives up, the error word reports MOE_ERR_DEVICE_TIMEOUT to the host, reading it clears it, and the
same context then runs a forward pass that matches the oracle."""
import numpy as np
import pytest
import torch

import nvfp4_expert_gemms_gb300 as M
import synth
from test_gpu_parity import Case, check_close

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = 5


def test_bounded_wait_timeout_is_reported_and_the_context_survives(orc):
    c = Case("fp8", 16, 256, 128, 8, 2, seed=21)
    c.run()  # sizes the workspace; the forward pass itself reports no error
    ws = c.layer.workspace
    M.moe_debug_wait_timeout(ws)
    assert M.moe_get_device_error(ws) == MOE_ERR_DEVICE_TIMEOUT
    assert M.moe_get_device_error(ws) == 0  # read and cleared
    got = synth.bf16_bits_to_f32(c.run())
    check_close(got, c.oracle(orc), "forward after a device timeout")


def test_wait_timeout_argument_errors():
    with pytest.raises(M.MoEError):
        M.moe_debug_wait_timeout(torch.empty(300, dtype=torch.uint8, device="cuda")[1:])
