"""Pins for the oracle's number-format codecs (CPU only).

Each codec is checked against something other than itself: PyTorch's own
float8_e4m3fn / bfloat16 casts (independent library implementations), the
bit-level definitions of the formats, hand-worked rounding cases, and a
second brute-force encoder that scans every code.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F


def brute_encode(t: float, table: np.ndarray, n_pos: int, sign_bit: int) -> int:
    """Scan all non-negative finite codes; nearest wins, ties go to the even code."""
    a = abs(float(t))
    best, best_d = 0, None
    for c in range(n_pos):
        d = abs(a - table[c])
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    if a >= table[n_pos - 1]:
        best = n_pos - 1
    return best | (sign_bit if np.signbit(t) else 0)


def test_e4m3_table_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ours = F.E4M3_TABLE
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.all(both_nan | (ref == ours))
    assert np.isnan(ours).sum() == 2            # 0x7F and 0xFF only
    assert np.signbit(ours[0x80]) and ours[0x80] == 0


def test_e4m3_spot_values():
    assert F.E4M3_TABLE[0x01] == 2.0 ** -9      # smallest subnormal
    assert F.E4M3_TABLE[0x07] == 7 * 2.0 ** -9
    assert F.E4M3_TABLE[0x08] == 2.0 ** -6      # smallest normal
    assert F.E4M3_TABLE[0x38] == 1.0
    assert F.E4M3_TABLE[0x7E] == 448.0
    assert F.E4M3_TABLE[0xFE] == -448.0


def test_e4m3_reencode_identity():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = F.E4M3_TABLE[codes].astype(np.float32)
    assert np.array_equal(F.e4m3_encode(vals), codes)


def test_e4m3_hand_rounding_cases():
    cases = {17.0: 0x58, 19.0: 0x5A, 2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02,
             -0.0: 0x80, 464.0: 0x7E, 449.0: 0x7E, 1e30: 0x7E, -1e30: 0xFE,
             float("inf"): 0x7E, float("-inf"): 0xFE, 7.5 * 2.0 ** -9: 0x08,
             432.0: 0x7E, 431.9: 0x7D}
    for t, c in cases.items():
        assert int(F.e4m3_encode(np.float32(t))) == c, (t, hex(c))
    assert int(F.e4m3_encode(np.float32("nan"))) == 0x7F


def test_e4m3_encode_matches_torch_in_range():
    g = np.random.Generator(np.random.PCG64(1))
    t = np.concatenate([
        g.standard_normal(200_000).astype(np.float32) * 100,
        (g.random(100_000) * 2 - 1).astype(np.float32) * 463.9,
        g.standard_normal(100_000).astype(np.float32) * 1e-2,
    ])
    # every midpoint between neighbours, and the float32 values either side of it
    mags = F.E4M3_TABLE[:0x7F]
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    t = np.concatenate([t, mids, -mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(t), ref)


def test_e4m3_encode_matches_brute_force():
    g = np.random.Generator(np.random.PCG64(2))
    t = np.concatenate([g.standard_normal(3000) * 50, g.standard_normal(500) * 1e-2,
                        g.standard_normal(200) * 1e4]).astype(np.float32)
    ours = F.e4m3_encode(t)
    for x, c in zip(t, ours):
        assert brute_encode(x, F.E4M3_TABLE, 0x7F, 0x80) == int(c)


def test_e2m1_table_and_ties():
    assert list(F.E2M1_TABLE[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(F.E2M1_TABLE[8:]) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
            6.5: 6.0, 100.0: 6.0, 0.24: 0.0, 0.26: 0.5, -5.01: -6.0, -0.0: -0.0}
    for t, v in ties.items():
        c = int(F.e2m1_encode(np.float32(t)))
        assert F.E2M1_TABLE[c] == v and np.signbit(F.E2M1_TABLE[c]) == np.signbit(v), (t, c)


def test_e2m1_encode_matches_brute_force():
    g = np.random.Generator(np.random.PCG64(3))
    t = (g.standard_normal(5000) * 3).astype(np.float32)
    ours = F.e2m1_encode(t)
    for x, c in zip(t, ours):
        assert brute_encode(x, F.E2M1_TABLE, 8, 0x8) == int(c)


def test_ue8m0_decode():
    assert F.ue8m0_decode(127) == 1.0
    assert F.ue8m0_decode(0) == 2.0 ** -127
    assert F.ue8m0_decode(254) == 2.0 ** 127
    assert np.isnan(F.ue8m0_decode(255))


def test_e2m1_packing_order():
    codes = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    packed = F.pack_e2m1(codes)
    assert packed.tolist() == [[0x21, 0x43]]          # element 2j in the low nibble
    assert np.array_equal(F.unpack_e2m1(packed), codes)


def test_round_to_bf16_matches_torch_on_float32_inputs():
    g = np.random.Generator(np.random.PCG64(4))
    x = np.concatenate([g.standard_normal(100_000) * 10.0 ** g.integers(-30, 30, 100_000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(F.round_to_bf16(x.astype(np.float64)), ref)


def test_round_to_bf16_single_rounding_from_float64():
    # 1 + 2^-8 + 2^-40 is just above the midpoint of 1 and 1 + 2^-7; a detour
    # through float32 would drop the 2^-40 and tie down to 1.0.
    assert F.round_to_bf16(1 + 2.0 ** -8 + 2.0 ** -40) == 1 + 2.0 ** -7
    assert F.round_to_bf16(1 + 2.0 ** -8) == 1.0                       # tie -> even
    assert F.round_to_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6          # tie -> even (up)
    assert F.round_to_bf16(-2.0 ** -140) == -0.0 or F.round_to_bf16(-2.0 ** -140) == 0
    assert F.round_to_bf16(3 * 2.0 ** -134) == 2 * 2.0 ** -133          # subnormal tie -> even
    assert np.isinf(F.round_to_bf16(2.0 ** 128))
    bits = F.f64_to_bf16_bits(np.array([1.0, -2.0, 0.1]))
    assert bits.tolist() == [0x3F80, 0xC000, 0x3DCD]
