"""The seeded input generator: published SplitMix64 values, determinism,
counter-mode slicing and the workloads' value ranges (no GPU)."""
import numpy as np

import synth


def test_splitmix64_published_sequence():
    """SplitMix64 from state 0 (Steele, Lea, Flood 2014; the reference
    implementation's first outputs)."""
    L = synth.lib()
    assert L.k3s_u64(0, 0) == 0xE220A8397B1DCDAF
    assert L.k3s_u64(0, 1) == 0x6E789E6AA1B965F4
    assert L.k3s_u64(0, 2) == 0x06C45D188009454F


def test_expert_planes_shapes_and_ranges():
    ex = synth.expert(1, 0, 5, d=256, f=64)
    assert ex["gate_packed"].shape == (64, 128) and ex["gate_scales"].shape == (64, 8)
    assert ex["down_packed"].shape == (256, 32) and ex["down_scales"].shape == (256, 2)
    for k in ["gate_scales", "up_scales", "down_scales"]:
        assert ex[k].min() >= 120 and ex[k].max() <= 130
    codes = np.concatenate([ex["gate_packed"].ravel() & 15, ex["gate_packed"].ravel() >> 4])
    hist = np.bincount(codes, minlength=16)
    assert hist.min() > 0.8 * codes.size / 16


def test_determinism_and_independence():
    a = synth.expert(1, 0, 5, d=128, f=32)
    b = synth.expert(1, 0, 5, d=128, f=32)
    c = synth.expert(1, 0, 6, d=128, f=32)
    assert np.array_equal(a["up_packed"], b["up_packed"])
    assert not np.array_equal(a["up_packed"], c["up_packed"])
    assert not np.array_equal(a["gate_packed"], a["up_packed"])


def test_counter_mode_prefix_property():
    """A stream's first n values do not depend on how many are drawn."""
    t = synth.tag(synth.K_MISC, 0, 0, 1)
    long = np.empty(1001, np.uint8)
    short = np.empty(77, np.uint8)
    synth.fill_bytes(long, t)
    synth.fill_bytes(short, t)
    assert np.array_equal(long[:77], short)
    x = synth.normal_f32((500,), t)
    y = synth.normal_f32((33,), t)
    assert np.array_equal(x[:33], y)


def test_normals_and_bf16():
    x = synth.token_f32(1, 0)
    assert x.dtype == np.float32 and x.shape == (7168,)
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1) < 0.05
    w = synth.router_bf16(1, 0, E=16, d=512)
    wf = (w.astype(np.uint32) << 16).view(np.float32)
    assert abs(wf.std() - 0.02) < 0.002
    # bf16 rounding of the same fp32 draws
    xf = synth.normal_f32((16, 512), synth.tag(synth.K_ROUTER, 1, 0), 0.0, 0.02)
    assert np.max(np.abs(wf - xf) / np.abs(xf)) <= 2.0 ** -8


def test_zipf_bias_is_log_rank():
    b = synth.bias_zipf(4, 0)
    r = np.sort(np.exp(-b.astype(np.float64) / 1.1))
    assert np.allclose(r, np.arange(1, 897), rtol=1e-5)
