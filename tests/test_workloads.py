"""Seeded input generators: determinism, layouts, dtype rounding (CPU only)."""
import numpy as np
import pytest

import workloads as W


def test_bf16_rounding_known_values():
    x = np.array([1.0, -2.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, 3.140625, 0.0],
                 dtype=np.float32)
    bits = W.f32_to_bf16_bits(x)
    # 1+2^-8 is a tie between 1.0 and 1+2^-7 -> even (1.0); 1+3*2^-8 -> 1+2^-6 (even)
    assert list(bits) == [0x3F80, 0xC000, 0x3F80, 0x3F82, 0x3F80, 0x4049, 0x0000]
    assert np.array_equal(W.bf16_bits_to_f32(bits)[:2], np.array([1.0, -2.0], dtype=np.float32))


def test_bf16_round_trip_is_identity_on_bf16_values():
    rng = np.random.default_rng(0)
    b = rng.integers(0, 0x7F80, 1000, dtype=np.uint16)  # finite positive bf16 patterns
    assert np.array_equal(W.f32_to_bf16_bits(W.bf16_bits_to_f32(b)), b)


@pytest.mark.parametrize("name", ["tiny_fp32", "decoder_bf16", "oddD_fp32"])
def test_deterministic_and_shaped(name):
    wl = W.WORKLOADS[name]
    if name != "tiny_fp32":
        wl = wl.with_(B=1, Q=7)
    a = W.make_inputs(wl)
    b = W.make_inputs(wl)
    for k in a:
        assert a[k].tobytes() == b[k].tobytes(), k
    B, S, M, D, L, K, Q = wl.B, wl.S, wl.M, wl.D, wl.L, wl.K, wl.Qn
    assert a["value"].shape == (B, S, M, D)
    assert a["sampling_locations"].shape == (B, Q, M, L, K, 2)
    assert a["attention_weights"].shape == (B, Q, M, L, K)
    assert a["grad_out"].shape == (B, Q, M * D)
    assert a["spatial_shapes"].dtype == np.int64 and a["spatial_shapes"].shape == (L, 2)
    assert list(a["level_start_index"]) == list(np.cumsum([0] + [h * w for h, w in wl.shapes])[:-1])
    attn = W.to_f64(a["attention_weights"], wl.dtype).reshape(-1, L * K)
    tol = {"f32": 1e-6, "f16": 1e-2, "bf16": 4e-2}[wl.dtype]
    assert np.allclose(attn.sum(-1), 1.0, atol=tol)
    loc = W.to_f64(a["sampling_locations"], wl.dtype)
    lo, hi = (-0.1, 1.1) if wl.loc == "uniform_wide" else (0.0, 1.0)
    assert loc.min() >= lo - 1e-6 and loc.max() <= hi + 1e-2


def test_encoder_reference_points():
    wl = W.WORKLOADS["encoder_fp16"].with_(B=1, shapes=((6, 10), (3, 5)))
    inp = W.make_inputs(wl)
    loc = W.to_f64(inp["sampling_locations"], "f16")
    assert loc.shape[1] == wl.S
    assert loc.min() >= -0.05 - 1e-3 and loc.max() <= 1.05 + 1e-3
    # query q = pixel q of the pyramid: the mean over (m, l, k) sits at its centre
    mean = loc.mean(axis=(2, 3, 4))[0]                    # [Q, 2]
    ref = W._pixel_centres(wl.shapes)
    assert np.abs(mean - ref).max() < 0.05


def test_full_size_metadata():
    st = W.WORKLOADS["stress_bf16"]
    assert st.S == 1044480 and st.B * st.S * st.M * st.D == 2139095040
    assert st.B * st.S * st.M * st.D * 2 > 2 ** 31          # byte offsets need 64 bits
    assert W.WORKLOADS["encoder_fp16"].Qn == 22223
    assert W.WORKLOADS["decoder_bf16"].units == 9600
