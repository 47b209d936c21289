"""Pins for the e4m3 input codec (sdpa_inputs.e4m3_encode / e4m3_decode),
which prepares the FP8 forward's inputs: against torch's float8_e4m3fn on
CPU, and against the format's definition at its edges."""
import numpy as np
import pytest

from sdpa_inputs import E4M3_MAX, e4m3_decode, e4m3_encode, quantize_e4m3


def test_decode_covers_the_format():
    vals = e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    finite = vals[np.isfinite(vals)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert e4m3_decode(np.array([1], dtype=np.uint8))[0] == 2.0 ** -9          # smallest subnormal
    assert e4m3_decode(np.array([8], dtype=np.uint8))[0] == 2.0 ** -6          # smallest normal
    assert e4m3_decode(np.array([0x38], dtype=np.uint8))[0] == 1.0
    # every non-NaN code round-trips
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = e4m3_encode(e4m3_decode(codes))
    ok = (back == codes) | ((codes == 0x80) & (back == 0x80))
    assert np.all(ok)


def test_encode_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    # exact ties between neighbouring codes (round half to even)
    grid = e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))
    ties = (grid[:-1] + grid[1:]) / 2
    x = np.concatenate([x, ties, -ties, [0.0, 448.0, -448.0, 2.0 ** -10, 3 * 2.0 ** -11]])
    x = x[np.abs(x) <= E4M3_MAX].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3_encode(x)
    np.testing.assert_array_equal(got, ref)


def test_saturation_and_quantisation():
    assert e4m3_encode(np.array([1000.0, -5000.0])).tolist() == [0x7E, 0xFE]   # +-448
    x = np.random.default_rng(1).standard_normal((4, 64)).astype(np.float32) * 3
    b, s = quantize_e4m3(x)
    deq = e4m3_decode(b) * s
    assert np.abs(deq).max() <= np.abs(x).max() * (1 + 1e-6)
    rel = np.abs(deq - x) / np.maximum(np.abs(x), 2.0 ** -6 * s)
    assert rel.max() <= 2.0 ** -4 + 1e-9        # half an ulp of a 3-bit mantissa
