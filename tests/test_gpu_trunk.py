"""The dense-trunk streamer's CUDA copier on the GPU: layers streamed through
the ring (and the resident prefix) arrive intact on the compute stream.
Each layer holds an expert blob; the expert GEMV on the streamed copy must
equal, bit for bit, the same kernel on a device-resident copy."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ring", [1, 2, 3])
def test_streamed_layers_arrive_intact(ring):
    d, f, M = 256, 256, 6
    eb = k.expert_bytes(d, f)
    host = torch.empty((M, eb), dtype=torch.uint8, pin_memory=True)
    dev = torch.empty((M, eb), dtype=torch.uint8, device="cuda")
    for l in range(M):
        planes = synth.expert(21, 0, l, d, f)
        for nm, arr in k.host_plane_views(host[l].data_ptr(), d, f).items():
            arr[...] = planes[nm]
    dev.copy_(host)
    x = torch.from_numpy(synth.token_f32(21, 0, d)).cuda()
    ws = torch.zeros(k.expert_gemv_workspace(d, f), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty_like(ws)
    pinned = 2 * ((eb + 255) // 256 * 256)  # layers 0 and 1 resident
    t = k.Trunk([host[l].data_ptr() for l in range(M)], [eb] * M, pinned, ring)
    s = k._stream()
    tokens = 3
    ys = torch.empty((tokens, M, d), dtype=torch.float32, device="cuda")
    ref = torch.empty((M, d), dtype=torch.float32, device="cuda")
    for l in range(M):
        k.expert_gemv(ref[l], x, k.expert_view(dev[l].data_ptr(), d, f), d, f, ws2)
    for tok in range(tokens):
        for l in range(M):
            p, resident, st = t.acquire(l, s)
            assert resident == (l < 2)
            k.expert_gemv(ys[tok, l], x, k.expert_view(p, d, f), d, f, ws)
            assert t.release(l, s) == 0
    torch.cuda.synchronize()
    assert k.device_error() == 0
    for tok in range(tokens):
        assert torch.equal(ys[tok], ref), tok
    st = t.stats()
    assert st["pinned_layers"] == 2 and st["resident"] == 2 * tokens
    assert st["prefetched"] == (tokens * (M - 2) if ring >= 2 else 0)
    t.close()
