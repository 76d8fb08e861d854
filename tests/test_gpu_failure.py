"""The failure path on the GPU, without a fault: a bounded wait that cannot complete
gives up after its limit, the host reads MOE_ERR_TIMEOUT from the device status word
(which the read clears), and the context stays usable for the layer afterwards."""
import time

import numpy as np
import pytest
import torch

import aux_loss_free_gb300 as M
from aux_loss_free_gb300.layer import LayerOnDevice, to_device_tokens
from synth import CONFIGS, make_layer

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 5


def test_bounded_wait_gives_up_and_reports():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    M.load_library()
    assert M.moe_device_status() == 0
    t0 = time.monotonic()
    assert M.moe_selftest_bounded_wait(2_000_000) == 1  # 2 ms limit
    assert time.monotonic() - t0 < 5.0
    assert M.moe_device_status() == MOE_ERR_TIMEOUT
    assert M.moe_device_status() == 0  # the read cleared it
    # The one-call form reports the same.
    assert M.moe_selftest_bounded_wait(1_000_000) == 1
    assert M.load_library().moe_last_device_status(None) == MOE_ERR_TIMEOUT
    assert M.load_library().moe_last_device_status(None) == 0
    # The context still runs the layer, and the same forward gives the same bits.
    s = CONFIGS["nano"].replace(T=256, d=256, E=16, f=128, F=128)
    host = make_layer(s, "nano")
    outs = []
    for _ in range(2):
        layer = LayerOnDevice(s, host, "cuda")
        out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device="cuda")
        layer.forward(to_device_tokens(host["x"], "cuda"), out, update_bias=False)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert np.isfinite(outs[0].float().cpu().numpy()).all()
    assert M.moe_device_status() == 0
