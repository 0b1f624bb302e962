"""Pins of the oracle's scalar arithmetic against libm, closed forms and an
independent brute-force E4M3 encoder (CPU only)."""
import math

import numpy as np
import pytest
import torch

import oracle


def _ulp32(y: np.ndarray) -> np.ndarray:
    """Spacing of binary32 numbers at |y| (for normal and subnormal y)."""
    a = np.abs(y).astype(np.float32)
    return (np.nextafter(a, np.float32(np.inf)) - a).astype(np.float64)


def test_exp_spec_closed_forms():
    assert oracle.exp_spec(0.0) == 1.0
    assert oracle.exp_spec(-100.0) == 0.0
    assert math.isinf(oracle.exp_spec(100.0))
    # exp(n ln2) = 2^n to within an ulp
    for n in range(-120, 120, 7):
        x = float(np.float32(n * math.log(2)))
        assert abs(oracle.exp_spec(x) - math.exp(x)) <= 1.0 * float(_ulp32(np.float32(math.exp(x))))


def test_exp_spec_vs_libm_sweep():
    x = np.linspace(-87.0, 88.0, 400_001, dtype=np.float32)
    x = np.concatenate([x, np.float32(-1.0) * np.logspace(-8, 0, 20_001, dtype=np.float32)])
    y = oracle.exp_spec_array(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    err = np.abs(y - ref) / _ulp32(ref.astype(np.float32))
    assert err.max() <= 2.0, err.max()


def test_tanh_spec_vs_libm_sweep():
    # every binary32 multiple of 2^-12 in [-1, 1] plus a dense sweep out to +-12
    x = np.concatenate([np.arange(-4096, 4097, dtype=np.float32) / np.float32(4096.0),
                        np.linspace(-12.0, 12.0, 300_001, dtype=np.float32),
                        np.logspace(-30, -1, 2001, dtype=np.float32)])
    y = oracle.tanh_spec_array(x).astype(np.float64)
    ref = np.tanh(x.astype(np.float64))
    err = np.abs(y - ref) / np.maximum(_ulp32(ref.astype(np.float32)), 1e-45)
    assert err.max() <= 4.0, err.max()
    # odd symmetry holds exactly; |t| >= 10 is exactly +-1
    assert np.array_equal(oracle.tanh_spec_array(-x), -y.astype(np.float32))
    assert oracle.tanh_spec(10.0) == 1.0 and oracle.tanh_spec(-37.5) == -1.0
    assert oracle.tanh_spec(0.0) == 0.0


def _torch_e4m3_table() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch_table():
    ours = oracle.e4m3_decode_table()
    ref = _torch_e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def _brute_e4m3(x: np.ndarray, mags: np.ndarray, codes: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 magnitude by search over the sorted code table;
    ties go to the even code; |x| beyond 448 saturates."""
    a = np.abs(x.astype(np.float64))
    i = np.clip(np.searchsorted(mags, a), 1, len(mags) - 1)
    lo, hi = mags[i - 1], mags[i]
    dlo, dhi = a - lo, hi - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[i] % 2 == 0))
    c = np.where(pick_hi, codes[i], codes[i - 1])
    c = np.where(a >= 448.0, 0x7E, c)
    return (c | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def test_e4m3_encode_exhaustive_binades():
    """Every positive binary32 in [2^-11, 2^9) (below: all round to zero;
    above: all saturate) against the brute-force nearest-code search; the
    negative half is checked on a strided subsample by sign symmetry."""
    table = oracle.e4m3_decode_table()
    pos = np.array([c for c in range(0x7F) if not np.isnan(table[c])])
    mags = table[pos]
    order = np.argsort(mags)
    mags, codes = mags[order], pos[order]
    for e in range(-11, 9):
        base = np.uint32((e + 127) << 23)
        x = (base + np.arange(1 << 23, dtype=np.uint32)).view(np.float32)
        got = oracle.e4m3_encode_array(x)
        assert np.array_equal(got, _brute_e4m3(x, mags, codes)), e
        neg = -x[::97]
        assert np.array_equal(oracle.e4m3_encode_array(neg), got[::97] | 0x80), e
    assert oracle.e4m3_encode(0.0) == 0x00 and oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(1e30) == 0x7E and oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(464.0) == 0x7E and oracle.e4m3_encode(2.0 ** -11) == 0x00


def test_e4m3_encode_vs_torch_cast():
    g = torch.Generator().manual_seed(1)
    x = (torch.randn(2_000_000, generator=g) * torch.exp(torch.randn(2_000_000, generator=g) * 3))
    x = x.clamp(-447.0, 447.0).to(torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_array(x.numpy())
    assert np.array_equal(got, ref)


def test_bf16_round_vs_torch():
    g = torch.Generator().manual_seed(2)
    x = (torch.randn(200_000, generator=g) * torch.exp(torch.randn(200_000, generator=g) * 8)).float()
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in x.numpy()], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # ties to even on exact binary32 midpoints
    assert oracle.bf16_round(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82


@pytest.mark.parametrize("bits", [0x3F800000, 0x00000001, 0x7F7FFFFF])
def test_bf16_round_edges(bits):
    v = float(np.uint32(bits).view(np.float32))
    ref = torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
    assert oracle.bf16_round(v) == ref
