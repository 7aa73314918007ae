"""The e4m3 weight format the fp8 workloads are drawn in (input generation,
shared by the oracle and the GPU path): pinned to the format's definition
(hand-decoded codes, ties to even, saturation, subnormals), to a library
conversion (torch.float8_e4m3fn), and the per-row quantisation's scale."""

import numpy as np
import pytest

import dflash2_synth as S


@pytest.mark.parametrize("x,code", [
    (448.0, 0x7E), (-448.0, 0xFE), (1.0, 0x38), (-1.5, 0xBC), (2.0, 0x40), (0.0, 0x00),
    (2.0 ** -6, 0x08),            # smallest normal
    (2.0 ** -9, 0x01),            # smallest subnormal
    (7 * 2.0 ** -9, 0x07),        # largest subnormal
    (1.0625, 0x38),               # tie between 1.0 and 1.125: to even mantissa 0
    (1.1875, 0x3A),               # tie between 1.125 and 1.25: to even mantissa 2
    (1.96875, 0x40),              # rounds up across the exponent boundary
    (2.0 ** -10, 0x00),           # tie between 0 and 2^-9: to even 0
    (3 * 2.0 ** -10, 0x02),       # tie between 1 and 2 (x 2^-9): to even 2
    (1000.0, 0x7E),               # saturates
])
def test_e4m3_codes_of_hand_values(x, code):
    assert int(S.e4m3_encode(np.array([x]))[0]) == code


def test_e4m3_decode_is_the_format_definition():
    # (1 + m/8) 2^(e-7) for e >= 1, m/8 2^-6 for e = 0, sign bit 7
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        v = S.e4m3_decode(np.array([c], dtype=np.uint8))[0]
        if e == 15 and m == 7:
            assert np.isnan(v)
            continue
        ref = (1 + m / 8) * 2.0 ** (e - 7) if e else m / 8 * 2.0 ** -6
        assert v == (-ref if s else ref)


def test_e4m3_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    np.testing.assert_array_equal(S.e4m3_encode(S.e4m3_decode(codes)), codes)


def test_e4m3_encode_matches_torch_float8():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    g = np.random.default_rng(0)
    x = np.concatenate([g.uniform(-448, 448, 100000), g.standard_normal(50000) * 0.01,
                        np.arange(-3000, 3000) * 2.0 ** -11])
    th = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(S.e4m3_encode(x), th)


def test_row_quantisation_scale_and_values():
    w = S._draw(5, "q", (64, 300), 0.02, "f32").values
    t = S.quantize_rows_e4m3(w)
    assert t.q.dtype == np.uint8 and t.scale.dtype == np.float32
    np.testing.assert_array_equal(t.scale, (np.max(np.abs(w), axis=1) / np.float32(448)).astype(np.float32))
    # each row's largest magnitude maps to +-448 exactly, and the values are q * scale
    assert np.all(np.max(np.abs(S.e4m3_decode(t.q)), axis=1) == 448.0)
    np.testing.assert_array_equal(t.values, S.e4m3_decode(t.q) * t.scale.astype(np.float64)[:, None])
    # relative error of e4m3 with 3 mantissa bits: at most 2^-4 of the value
    # for normals, 2^-10 * scale absolute in the subnormal range
    err = np.abs(t.values - w)
    assert np.all(err <= np.maximum(np.abs(w) * 2.0 ** -4, 2.0 ** -10 * t.scale[:, None]) + 1e-12)


def test_target_probs_truncation():
    # the synthetic target distributions: each row sums to 1, keeps at most
    # top_k tokens, and its kept set is the smallest prefix (in probability
    # order) whose mass reaches top_p
    p = S.make_target_probs(50, 300, seed=3, top_p=0.9, top_k=20)
    assert p.dtype == np.float32 and p.shape == (50, 300)
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-5)
    for row in p.astype(np.float64):
        kept = np.sort(row[row > 0])[::-1]
        assert 1 <= kept.size <= 20
        # dropping the smallest kept token would leave less than top_p of the
        # (top-k renormalised) mass, so it had to stay
        assert np.all(np.diff(kept) <= 1e-12)
