"""A bounded wait that runs out ends in an error status, not a hung GPU: a
kernel waits on a barrier nothing completes, gives up after its limit, the
host reads K3MOE_ETIMEOUT, and the context keeps working."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import rel_err
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


def test_wait_on_nothing_times_out_and_the_context_survives():
    assert k.device_error() == 0
    t0 = time.time()
    k.check_wait_timeout()
    assert k.device_error() == k.K3MOE_ETIMEOUT
    assert 1.5 < time.time() - t0 < 30
    assert k.device_error() == 0  # read-and-clear
    # the context still runs kernels correctly
    d, f = 512, 256
    ex = synth.expert(31, 0, 0, d, f)
    blob = torch.empty(k.expert_bytes(d, f), dtype=torch.uint8, device="cuda")
    k.pack_expert(blob, ex, d, f)
    x = synth.token_f32(31, 0, d)
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    ws = torch.zeros(k.expert_gemv_workspace(d, f) // 4 + 4, dtype=torch.float32, device="cuda")
    k.expert_gemv(y, torch.from_numpy(x).cuda(), k.expert_view(blob.data_ptr(), d, f), d, f, ws)
    torch.cuda.synchronize()
    assert rel_err(y.cpu().numpy(), oracle.expert_forward(ex, x)) <= 2e-3
    assert k.device_error() == 0
