"""The allocation-free single-expert entry point, k3moe_expert_gemv_noalloc.

It serves callers that may not allocate device memory on the call path (for
example code running inside a global-mode stream capture, or a thread with a
no-allocation rule): its scratch is a fixed device array inside the library.
Here it is checked, through the C ABI, against the fp64 oracle and against
k3moe_expert_gemv (which takes a caller-allocated workspace) on two calls in
a row, so the second call also shows that the shared scratch left by the
first does not leak into it.  The file is named to run last.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import TOL, rel_err
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


def _planes(e, d, f):
    return synth.expert(11, 0, e, d, f)


def _blob(planes, d, f):
    blob = torch.empty(k.expert_bytes(d, f), dtype=torch.uint8, device="cuda")
    keep = k.pack_expert(blob, planes, d, f)
    torch.cuda.synchronize()
    del keep
    return blob


@pytest.mark.parametrize("d,f", [(7168, 1536), (1056, 544), (7168, k.K3MOE_NOALLOC_MAX_F)])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(d, f):
    planes = [_planes(e, d, f) for e in range(2)]
    blobs = [_blob(p, d, f) for p in planes]
    views = [k.expert_view(b.data_ptr(), d, f) for b in blobs]
    ws = torch.zeros(k.expert_gemv_workspace(d, f) // 4, dtype=torch.float32, device="cuda")
    for call in range(2):
        x = synth.token_f32(11, call, d)
        xd = torch.from_numpy(x).cuda()
        y_ref = torch.empty(d, dtype=torch.float32, device="cuda")
        y_na = torch.full((d,), float("nan"), dtype=torch.float32, device="cuda")
        k.expert_gemv(y_ref, xd, views[call], d, f, ws)
        k.expert_gemv_noalloc(y_na, xd, views[call], d, f)
        torch.cuda.synchronize()
        a, b = y_na.cpu().numpy(), y_ref.cpu().numpy()
        assert np.all(np.isfinite(a))
        ref = oracle.expert_forward(planes[call], x.astype(np.float64))
        assert rel_err(a, ref) <= TOL, (call, rel_err(a, ref))
        assert rel_err(a, b) <= TOL, (call, rel_err(a, b))
    assert k.device_error() == 0


def test_noalloc_takes_no_device_memory():
    """After a first call (which loads the kernels and looks up the scratch
    address), further calls leave the device's free memory unchanged."""
    d, f = 1056, 544
    blob = _blob(_planes(0, d, f), d, f)
    view = k.expert_view(blob.data_ptr(), d, f)
    x = torch.from_numpy(synth.token_f32(11, 0, d)).cuda()
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    k.expert_gemv_noalloc(y, x, view, d, f)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        k.expert_gemv_noalloc(y, x, view, d, f)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_reports_through_the_device_error_word():
    """The entry point shares the one device error word that
    k3moe_device_error() reads: a timeout recorded by the bounded-wait
    self-check is still there after noalloc calls (they neither clear it nor
    use another word), is read once, and is then cleared."""
    d, f = 1056, 544
    blob = _blob(_planes(1, d, f), d, f)
    view = k.expert_view(blob.data_ptr(), d, f)
    x = torch.from_numpy(synth.token_f32(11, 1, d)).cuda()
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    assert k.device_error() == 0
    k.check_wait_timeout()
    k.expert_gemv_noalloc(y, x, view, d, f)
    assert k.device_error() == k.K3MOE_ETIMEOUT
    assert k.device_error() == 0


def test_noalloc_refuses_sizes_beyond_its_scratch():
    d, f = 1024, k.K3MOE_NOALLOC_MAX_F + 32
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    x = torch.zeros(d, dtype=torch.float32, device="cuda")
    e = k.expert_view(1 << 20, d, f)  # never dereferenced: the size check comes first
    with pytest.raises(k.K3Error) as ei:
        k.expert_gemv_noalloc(y, x, e, d, f)
    assert ei.value.status == k.K3MOE_EINVAL
