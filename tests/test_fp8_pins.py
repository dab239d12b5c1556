"""Pins of the oracle's FP8 E4M3 codec, the element format an FP8 KV cache
would use (reading: OCP E4M3 without infinities, round to nearest with ties
to the even code, saturation to +-448).  Independent of the oracle's C code:
PyTorch's own float8_e4m3fn conversion (a library routine), closed-form
special values, and round trips."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
if not hasattr(torch, "float8_e4m3fn"):
    pytest.skip("this PyTorch has no float8_e4m3fn", allow_module_level=True)


def _library_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_of_every_code_matches_the_library():
    mine = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = _library_decode_all()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S 1111 111
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_encode_matches_the_library_in_range_including_ties():
    table = _library_decode_all()
    mags = np.unique(np.abs(table[~np.isnan(table)]))          # 0 .. 448
    mids = (mags[:-1] + mags[1:]) / 2                           # exact ties (5 significant bits)
    rng = np.random.default_rng(0)
    rand = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.02, 1.0, 30.0, 200.0)])
    x = np.concatenate([rand, mags, mids, -mags, -mids]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = oracle.e4m3_encode(x.astype(np.float64))
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(mine[i]), int(ref[i])) for i in bad[:5]]


def test_special_values_and_saturation():
    enc = lambda v: int(oracle.e4m3_encode(np.array([v]))[0])
    assert enc(1.0) == 0x38 and enc(-2.0) == 0xC0 and enc(448.0) == 0x7E
    for v in (449.0, 463.9, 464.0, 1e9, np.inf):  # finite overflow and infinity saturate
        assert enc(v) == 0x7E and enc(-v) == 0xFE
    assert enc(np.nan) & 0x7F == 0x7F
    assert enc(0.0) == 0x00 and enc(-0.0) == 0x80
    assert enc(2.0 ** -9) == 0x01          # smallest subnormal
    assert enc(2.0 ** -10) == 0x00         # tie between 0 and 2^-9: the even code
    assert enc(3 * 2.0 ** -10) == 0x02     # tie between 2^-9 and 2^-8: the even code
    assert enc(0.96875) == 0x38            # tie between 0.9375 (0x37) and 1.0 (0x38)


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)
