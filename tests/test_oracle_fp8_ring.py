"""Pins for the oracle's E4M3 codec, absmax quantiser and list ring (CPU only).

The codec is pinned to the OCP FP8 specification's printed values
(tests/golden/e4m3_ocp_values.txt), to PyTorch's float8_e4m3fn conversion
(a library routine, round-to-nearest-even) wherever no saturation is involved,
and to exhaustive round trips and tie cases.  The ring is pinned to the
closed form "the last R chunks are held, chunk c in slot c mod R".
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import fp8
from oracle.ring import ListRing, RingError, expected_physical_slots, slot_of

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_ocp_table():
    with open(os.path.join(GOLDEN, "e4m3_ocp_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            code, val = line.split()
            got = fp8.e4m3_decode_code(int(code, 16))
            if val == "nan":
                assert math.isnan(got)
            else:
                assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_decode_all_codes_matches_torch():
    ours = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = _torch_decode_all()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.sum(np.isnan(ours)) == 2


def test_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = fp8.e4m3_decode(codes).astype(np.float32)
    back = fp8.e4m3_encode(vals)
    assert np.array_equal(back, codes)


def test_midpoints_round_to_even_and_neighbours():
    pos = fp8.e4m3_decode(np.arange(127, dtype=np.uint8))
    for c in range(126):
        mid = np.float32((pos[c] + pos[c + 1]) / 2)  # exact: needs 5 significant bits
        assert float(mid) == (pos[c] + pos[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert fp8.e4m3_encode(np.array([mid]))[0] == want
        assert fp8.e4m3_encode(np.array([-mid]))[0] == (want | 0x80)
        up = np.nextafter(mid, np.float32(np.inf), dtype=np.float32)
        dn = np.nextafter(mid, np.float32(-np.inf), dtype=np.float32)
        assert fp8.e4m3_encode(np.array([up]))[0] == c + 1
        assert fp8.e4m3_encode(np.array([dn]))[0] == c


def test_saturation_and_special():
    x = np.array([448.0, 449.0, 463.99, 464.0, 1e6, np.inf, -500.0, -np.inf], dtype=np.float32)
    assert list(fp8.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert fp8.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F
    tiny = np.array([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11), 2.0 ** -10, 1.5 * 2.0 ** -10], np.float32)
    # 2^-11 rounds to 0 (keeps sign); 2^-10 is the tie between 0 and 2^-9 -> even (0);
    # 1.5*2^-10 is above the tie -> 2^-9 (code 1)
    assert list(fp8.e4m3_encode(tiny)) == [0x00, 0x80, 0x00, 0x80, 0x00, 0x01]


def test_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.normal(size=200_000).astype(np.float32) * 100,
        rng.uniform(-448, 448, size=200_000).astype(np.float32),
        (rng.normal(size=100_000) * 2.0 ** -8).astype(np.float32),
    ])
    x = x[np.abs(x) <= 448]
    ours = fp8.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_quantize_block_properties():
    rng = np.random.default_rng(1)
    x = (rng.normal(size=(405, 128)) * np.where(rng.random((405, 128)) < 0.01, 8, 1)).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    codes, s = fp8.quantize_block(x)
    amax = np.float32(np.abs(x).max())
    assert s == np.float32(amax / np.float32(448.0))
    assert int((codes & 0x7F).max()) == 0x7E  # the absmax element maps to 448
    xh = fp8.dequantize_block(codes, s)
    vals = np.abs(x / np.float64(s))
    # half-ulp bound of E4M3: 2^-4 relative for normals, 2^-10 absolute below 2^-6
    bound = np.where(vals >= 2.0 ** -6, vals * 2.0 ** -4, 2.0 ** -10) * np.float64(s) * (1 + 1e-6)
    assert np.all(np.abs(xh - x) <= bound + np.abs(x) * 2.0 ** -23)


def test_quantize_zero_block():
    codes, s = fp8.quantize_block(np.zeros((4, 8), np.float32))
    assert s == np.float32(1.0) and np.all(codes == 0)


def test_quantize_chunk_layout():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(2, 5, 3, 8)).astype(np.float32)
    codes, scales = fp8.quantize_chunk_bhld(x)
    assert codes.shape == (2, 3, 5, 8) and scales.shape == (2, 3)
    c, s = fp8.quantize_block(x[1, :, 2, :])
    assert np.array_equal(codes[1, 2], c) and scales[1, 2] == s


@pytest.mark.parametrize("R", [1, 2, 3, 20])
def test_ring_holds_last_R_and_slot_mapping(R):
    ring = ListRing(R)
    phys = np.full((R,), -1)
    for c in range(3 * R + 1):
        ring.append(c, np.array([c]), np.array([-c]))
        phys[slot_of(c, R)] = c
        assert ring.held_chunks() == list(range(max(0, c - R + 1), c + 1))
        held_slots = sorted(slot_of(x, R) for x in ring.held_chunks())
        assert held_slots == sorted(set(held_slots))  # distinct slots
        exp = expected_physical_slots(ring, np.full((R, 1), -1), 0)[:, 0]
        for x in ring.held_chunks():
            assert exp[slot_of(x, R)] == x == phys[slot_of(x, R)]
        if c < R - 1:  # never-written slots keep the initial value
            assert np.all(exp[c + 1:] == -1)


def test_ring_rewrite_and_order_errors():
    ring = ListRing(2)
    ring.append(0, np.array([1]), np.array([1]))
    ring.append(0, np.array([2]), np.array([2]))  # rewrite of the newest chunk
    assert ring.held_chunks() == [0] and ring.get(0)[0][0] == 2
    ring.append(1, np.array([3]), np.array([3]))
    with pytest.raises(RingError):
        ring.append(3, np.array([0]), np.array([0]))
    with pytest.raises(RingError):
        ring.append(0, np.array([0]), np.array([0]))
    with pytest.raises(RingError):
        ring.get(5)
