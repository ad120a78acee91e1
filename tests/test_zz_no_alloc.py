"""The allocation-free single-expert entry point, k3moe_expert_gemv_noalloc.

It serves callers that may not allocate device memory on the call path (for
example code running inside a global-mode stream capture, or a thread with a
no-allocation rule): its scratch is a fixed device array inside the library.
Here it is checked, through the C ABI, against k3moe_expert_gemv (which takes
a caller-allocated workspace) on two calls in a row, so the second call also
shows that the shared scratch left by the first does not leak into it.  The
file is named to run last.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import TOL, rel_err
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


def _blob(pool, e, d, f):
    blob = torch.empty(k.expert_bytes(d, f), dtype=torch.uint8, device="cuda")
    keep = k.pack_expert(blob, synth.expert(pool, 0, e, d, f), d, f)
    torch.cuda.synchronize()
    del keep
    return blob


@pytest.mark.parametrize("d,f", [(7168, 1536), (1056, 544)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(d, f):
    blobs = [_blob(11, e, d, f) for e in range(2)]
    views = [k.expert_view(b.data_ptr(), d, f) for b in blobs]
    ws = torch.empty(k.expert_gemv_workspace(d, f) // 4, dtype=torch.float32, device="cuda")
    for call in range(2):
        x = torch.from_numpy(synth.token_f32(11, call, d)).cuda()
        y_ref = torch.empty(d, dtype=torch.float32, device="cuda")
        y_na = torch.full((d,), float("nan"), dtype=torch.float32, device="cuda")
        k.expert_gemv(y_ref, x, views[call], d, f, ws)
        k.expert_gemv_noalloc(y_na, x, views[call], d, f)
        torch.cuda.synchronize()
        a, b = y_na.cpu().numpy(), y_ref.cpu().numpy()
        assert np.all(np.isfinite(a))
        assert rel_err(a, b) <= TOL, (call, rel_err(a, b))


def test_noalloc_refuses_sizes_beyond_its_scratch():
    d, f = 1024, k.K3MOE_NOALLOC_MAX_F + 32
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    x = torch.zeros(d, dtype=torch.float32, device="cuda")
    e = k.expert_view(1 << 20, d, f)  # never dereferenced: the size check comes first
    with pytest.raises(k.K3Error) as ei:
        k.expert_gemv_noalloc(y, x, e, d, f)
    assert ei.value.status == k.K3MOE_EINVAL
