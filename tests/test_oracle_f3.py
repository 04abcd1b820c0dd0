"""Pins for the oracle's native base-3 packing (no GPU).

The card gives the information content of a trit (log2 3 bits) and the 1.71
bits/weight it implies with the FP16 scale, and names packing at that density
as future work ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card, "Weight
representation: ternary g128" and "Memory requirement"); it gives no layout.
The layout read here: five trits per byte (q0 + 3 q1 + 9 q2 + 27 q3 + 81 q4,
q = t + 1), 25 such bytes and a three-trit 26th per 128-weight group.

The pins check the oracle against things other than itself: every five-trit
and three-trit pattern (a bijection onto 0..242 and 0..26, and the round
trip), a hand-worked byte, out-of-range detection, the dense product from an
explicitly expanded W and the 2-bit oracle on the same trits, and the card's
bit-rate figures.
"""
import json
import math
import os

import numpy as np

import synth
from tests.test_oracle import bf16_bits_to_f64, dense_w

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_every_five_trit_pattern_is_one_byte(orc):
    """All 3^5 patterns at a group's first five positions: 243 distinct bytes
    0..242, each unpacking to its pattern; likewise the 3^3 patterns of the
    group's last byte (trits 125..127) give 27 distinct bytes 0..26."""
    pats = np.array(np.meshgrid(*[[-1, 0, 1]] * 5, indexing="ij")).reshape(5, -1).T   # [243, 5]
    t = np.zeros((243, 128), dtype=np.int8)
    t[:, 0:5] = pats
    packed, bad = orc.f3_pack(t)
    assert bad == 0 and packed.shape == (243, 26)
    assert sorted(packed[:, 0].tolist()) == list(range(243))
    back, bad = orc.f3_unpack(packed, 128)
    assert bad == 0 and np.array_equal(back, t)
    pats3 = np.array(np.meshgrid(*[[-1, 0, 1]] * 3, indexing="ij")).reshape(3, -1).T  # [27, 3]
    t3 = np.zeros((27, 128), dtype=np.int8)
    t3[:, 125:128] = pats3
    packed3, bad = orc.f3_pack(t3)
    assert bad == 0
    assert sorted(packed3[:, 25].tolist()) == list(range(27))
    back3, _ = orc.f3_unpack(packed3, 128)
    assert np.array_equal(back3, t3)


def test_hand_worked_byte():
    """t = (1, 0, -1, 0, 1) at positions 0..4: q = (2, 1, 0, 1, 2), byte
    2 + 3 + 0 + 27 + 162 = 194; position 5 starts the next byte."""
    import oracle
    t = np.zeros((1, 128), dtype=np.int8)
    t[0, :5] = [1, 0, -1, 0, 1]
    t[0, 5] = 1
    packed, _ = oracle.f3_pack(t)
    assert packed[0, 0] == 194
    assert packed[0, 1] == 2 + 1 * 3 + 1 * 9 + 1 * 27 + 1 * 81   # q = 2 then four zeros (q = 1)
    assert packed[0, 25] == 1 + 3 + 9                             # trits 125..127 all zero


def test_round_trip_and_invalid_entries(orc):
    t = synth.trits(70, "f3rt", (37, 1024))
    packed, bad = orc.f3_pack(t)
    assert bad == 0
    back, bad = orc.f3_unpack(packed, 1024)
    assert bad == 0 and np.array_equal(back, t)
    t2 = t.copy()
    t2[3, 17] = 2
    t2[9, 1000] = -5
    _, bad = orc.f3_pack(t2)
    assert bad == 2
    p2 = packed.copy()
    p2[0, 0] = 243            # not a five-trit byte
    p2[1, 25] = 27            # not a three-trit byte
    p2[2, 24] = 242           # the largest valid byte
    _, bad = orc.f3_unpack(p2, 1024)
    assert bad == 2


def test_product_matches_dense_and_two_bit_oracle(orc):
    """The base-3 product equals the dense product of the expanded W (up to
    fp64 rounding order) and the 2-bit oracle's product on the same trits."""
    M, N, K = 3, 41, 640
    p = synth.problem(71, M, N, K, tag="f3dense")
    packed, bad = orc.f3_pack(p.t)
    assert bad == 0
    y, a = orc.f3_matmul(p.x, packed, p.s)
    x = bf16_bits_to_f64(p.x)
    w = dense_w(p.t, p.s.astype(np.float64))
    y_dense = x @ w.T
    a_dense = np.abs(x) @ np.abs(w).T
    assert np.allclose(y, y_dense, rtol=1e-12, atol=1e-12 * a_dense.max())
    assert np.allclose(a, a_dense, rtol=1e-12)
    codes, _ = orc.pack(p.t)
    y2, a2 = orc.matmul(p.x, codes, p.s)
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-12 * a2.max())


def test_bit_rate_against_the_card():
    """26 bytes per 128 weights plus the FP16 scale: 1.75 bits/weight, between
    the card's theoretical 1.71 (log2 3 + 16/128) and the deployed 2.125, and
    18 % fewer bytes than the 2-bit slots."""
    g = json.load(open(os.path.join(GOLDEN, "bitrates.json")))
    bpw = (26 * 8 + 16) / 128
    assert bpw == 1.75
    theo = math.log2(3) + 16 / 128
    assert round(theo, 2) == g["theoretical_bpw"]["value"]
    assert g["theoretical_bpw"]["value"] < bpw < g["deployed_bpw"]["value"]
    assert (bpw - theo) / theo < 0.025
    assert abs(1 - bpw / g["deployed_bpw"]["value"] - 0.176) < 0.001
    # five trits fit a byte (3^5 = 243 <= 256), six do not
    assert 3 ** 5 <= 256 < 3 ** 6
