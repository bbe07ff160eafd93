"""Pins of the oracle's FP8 (E4M3) storage of the Mean-K index.

The codec is checked against facts of the E4M3 format that do not restate the
oracle's formula: landmark values, the count and order of the finite values,
nearest-value rounding by brute force over all 254 finite codes, the even-code
rule on ties, round trips.  The per-row scale is checked for minimality by
brute force, and the stored values for exactness in bf16.  Hand-worked rows
pin the whole path.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle


def _finite_codes():
    return [c for c in range(256) if not math.isnan(oracle.e4m3_decode(c))]


def test_e4m3_landmarks():
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x7E) == 448.0            # largest finite
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6        # smallest normal
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9        # smallest subnormal
    assert oracle.e4m3_decode(0x00) == 0.0 and math.copysign(1, oracle.e4m3_decode(0x80)) < 0
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    assert oracle.e4m3_decode(0xB8) == -1.0


def test_e4m3_value_set():
    fin = _finite_codes()
    assert len(fin) == 254                              # 256 codes minus the two NaNs
    pos = [oracle.e4m3_decode(c) for c in range(0x00, 0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))      # codes 0x00..0x7E ascend
    for c in range(0x80):
        if c != 0x7F:
            assert oracle.e4m3_decode(c | 0x80) == -oracle.e4m3_decode(c)
    # 3 mantissa bits: 8 values per binade, evenly spaced, from 2^-6 to 2^8
    for E in range(-6, 9):
        vals = [v for v in pos if 2.0 ** E <= v < 2.0 ** (E + 1)]
        assert len(vals) == (7 if E == 8 else 8)
        assert len({b - a for a, b in zip(vals, vals[1:])}) == 1


def test_e4m3_encode_is_nearest_with_ties_to_even():
    fin = _finite_codes()
    table = np.array([oracle.e4m3_decode(c) for c in fin])
    rng = np.random.default_rng(0)
    ys = np.concatenate([rng.uniform(-448, 448, 3000), rng.uniform(-0.05, 0.05, 2000),
                         [0.0, 448.0, -448.0, 2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875, 464.0 - 1e-9]])
    ys = ys[np.abs(ys) <= 448]
    for y in ys:
        c = oracle.e4m3_encode(y)
        v = oracle.e4m3_decode(c)
        d = np.abs(table - y)
        best = d.min()
        assert abs(v - y) == best, (y, hex(c))
        ties = [fin[i] for i in np.flatnonzero(d == best)]
        if len({oracle.e4m3_decode(t) for t in ties}) > 1:   # a true tie between two values
            assert (c & 1) == 0, (y, hex(c))
        assert (c & 0x80) == (0x80 if math.copysign(1.0, y) < 0 else 0)
    # round trip of every finite code
    for c in fin:
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c


@pytest.mark.parametrize("seed", range(4))
def test_fp8_row_exp_is_minimal(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        x = rng.standard_normal(16) * 10.0 ** rng.uniform(-20, 20)
        e = oracle.fp8_row_exp(x)
        m = np.abs(x).max()
        assert m <= 448 * 2.0 ** e
        assert e == -100 or m > 448 * 2.0 ** (e - 1)
    assert oracle.fp8_row_exp(np.zeros(8)) == -100
    assert oracle.fp8_row_exp(np.array([448.0])) == 0 and oracle.fp8_row_exp(np.array([448.5])) == 1
    assert oracle.fp8_row_exp(np.array([224.0])) == -1 and oracle.fp8_row_exp(np.array([1e-40])) == -100


def _bits(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_index_fp8_hand_worked_rows():
    # max 300: 300 = 0.586 * 2^9, so e = 0; 300 / 2^5 = 9.375 -> code 0x79 (288); -0.1 -> 13/128 (0x9D)
    # max 1000 = 0.977 * 2^10, so e = 2: 1000/4 = 250 rounds up a binade to 256 (0x78); 1/4 -> 0x28
    rows = np.array([[1.0, -0.1, 300.0, 0.0], [1000.0, 1.0, 0.0, -0.0]])
    codes, exps = oracle.index_to_fp8(_bits(rows))
    assert exps.tolist() == [0, 2]
    assert codes.tolist() == [[0x38, 0x9D, 0x79, 0x00], [0x78, 0x28, 0x00, 0x80]]
    back = oracle.bf16_to_f64(oracle.index_from_fp8(codes, exps))
    assert back.tolist() == [[1.0, -0.1015625, 288.0, 0.0], [1024.0, 1.0, 0.0, -0.0]]


@pytest.mark.parametrize("seed", range(3))
def test_index_fp8_round_trip_bounds(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((64, 128)) * 10.0 ** rng.uniform(-8, 8, (64, 1))
    x[3] = 0.0
    b = _bits(x)
    codes, exps = oracle.index_to_fp8(b)
    back_bits = oracle.index_from_fp8(codes, exps)
    xv, back = oracle.bf16_to_f64(b), oracle.bf16_to_f64(back_bits)
    # every stored value is code * 2^e exactly, and exact in bf16
    dec = np.vectorize(oracle.e4m3_decode)(codes) * 2.0 ** exps[:, None].astype(np.float64)
    assert np.array_equal(back, dec)
    # relative error at most half a step (2^-4) where the scaled value is normal in E4M3
    scaled = np.abs(xv) * 2.0 ** (-exps[:, None].astype(np.float64))
    normal = scaled >= 2.0 ** -6
    assert np.all(np.abs(back - xv)[normal] <= 2.0 ** -4 * np.abs(xv)[normal])
    # below that, at most half the subnormal step 2^-9 (scaled)
    assert np.all((np.abs(back - xv) * 2.0 ** (-exps[:, None].astype(np.float64)))[~normal] <= 2.0 ** -10)
    # the largest element of each nonzero row lands in the top binade of the format
    nz = np.abs(xv).max(axis=1) > 0
    top = (np.abs(xv).max(axis=1) * 2.0 ** (-exps.astype(np.float64)))[nz]
    assert np.all((top > 224) & (top <= 448))
    # quantising stored values again stores the same values (a row whose maximum rounded
    # down to 224 may now take the next smaller exponent, with codes one binade up)
    c2, e2 = oracle.index_to_fp8(back_bits)
    assert np.array_equal(oracle.index_from_fp8(c2, e2), back_bits)
    assert np.all((e2 == exps) | (e2 == exps - 1))
