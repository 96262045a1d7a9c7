"""Pins of the oracle's FP8 E4M3 KV storage (CPU only).

The format is the OCP 8-bit floating point E4M3 ("E4M3FN"): its codes and
their values are checked against PyTorch's float8_e4m3fn conversion (a
library routine), and the saturating limit against the format's closed
form.  The quantized store of the oracle is checked against a model built
from that library conversion: quantize every row with torch, run the plain
fp64 oracle on the dequantized rows, and require the same outputs and skip
sets bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle.oracle import OracleStream, e4m3_decode, e4m3_encode

E4M3_MAX = 448.0          # 1.75 * 2^8
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9


def torch_codes(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_matches_the_library_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([e4m3_decode(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.isnan(got).sum() == 2  # 0x7F and 0xFF only
    assert got[0x7E] == E4M3_MAX and got[0x08] == E4M3_MIN_NORMAL and got[0x01] == E4M3_MIN_SUBNORMAL


def _in_range_values(rng):
    finite = np.array([e4m3_decode(c) for c in range(127)])
    mids = (finite[:-1] + finite[1:]) / 2  # exact midpoints: ties
    near = np.concatenate([np.nextafter(mids.astype(np.float32), np.float32(0)),
                           np.nextafter(mids.astype(np.float32), np.float32(1e9))])
    rand = np.ldexp(rng.uniform(1, 2, 4000), rng.integers(-14, 9, 4000))
    vals = np.concatenate([finite, mids, near, rand, [464.0, 463.99, 1e-30, 0.0]]).astype(np.float32)
    vals = vals[np.abs(vals) <= 464.0]
    return np.concatenate([vals, -vals])


def test_encode_matches_the_library_in_range():
    vals = _in_range_values(np.random.default_rng(11))
    got = np.array([e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, torch_codes(vals))


def test_encode_saturates_beyond_the_largest_finite_value():
    for v in (464.5, 480.0, 1e6, float("inf")):
        assert e4m3_encode(v) == 0x7E and e4m3_encode(-v) == 0xFE
    assert e4m3_encode(float("nan")) & 0x7F == 0x7F


def test_quantized_store_equals_the_library_model():
    """The bit-exact check of the E4M3 store (registered as the fp8_store
    pin, so planted storage mistakes are shown to fail it)."""
    from tests import pins

    assert not pins.pin_fp8_store()


def test_quantized_store_is_the_identity_on_representable_rows():
    """Rows whose elements are E4M3 values times a power-of-two scale are
    stored exactly, so the FP8 oracle equals the plain one."""
    rng = np.random.default_rng(9)
    finite = np.array([e4m3_decode(c) for c in range(127)] + [-e4m3_decode(c) for c in range(1, 127)])
    d, L_p, L_dec, N_r, N_att = 8, 5, 30, 12, 5
    scale = 2.0 ** -5
    pick = lambda *shape: rng.choice(finite, shape) * scale
    K, V, k, v = pick(L_p, d), pick(L_p, d), pick(L_dec, d), pick(L_dec, d)
    q = rng.normal(0, 1, (L_dec, d))
    a = OracleStream(d, L_p, N_r, N_att, 0, kv_scales=(scale, scale))
    b = OracleStream(d, L_p, N_r, N_att, 0)
    a.prefill(K, V)
    b.prefill(K, V)
    for t in range(L_dec):
        oa, _ = a.step(q[t], k[t], v[t])
        ob, _ = b.step(q[t], k[t], v[t])
        assert np.array_equal(oa, ob)


def test_quantization_error_is_within_half_a_step():
    """|stored - x| <= 2^-4 |x| in the normal range (3 mantissa bits, round
    to nearest) and <= 2^-10 * scale in the subnormal range."""
    rng = np.random.default_rng(3)
    d, scale = 64, 0.05  # |x| / scale stays below 448: no saturation
    x = np.concatenate([np.clip(rng.normal(0, 3, d // 2), -20, 20), rng.uniform(-1e-4, 1e-4, d // 2)])
    s = OracleStream(d, 1, 4, 2, 0, kv_scales=(scale, scale))
    s.prefill(x[None, :], x[None, :])
    out, _ = s.step(np.zeros(d), x, x)  # q = 0: uniform weights over the prompt row and the new row
    stored = out  # both rows equal, so the output is the stored row
    y = np.abs(x) / scale
    bound = np.where(y >= E4M3_MIN_NORMAL, 2.0 ** -4 * np.abs(x), 2.0 ** -10 * scale)
    assert (np.abs(stored - x) <= bound * (1 + 1e-12)).all()


def test_scales_must_be_positive_and_finite():
    for bad in ((0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0), (1.0, float("nan"))):
        with pytest.raises(ValueError):
            OracleStream(8, 1, 4, 2, 0, kv_scales=bad)
