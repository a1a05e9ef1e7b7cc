"""Pins of the BF16 bit-field oracle: hand-derived fields, the IEEE value formula, and
exhaustive round trips.  CPU only."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import bitfield_oracle as B

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    return json.load(open(os.path.join(HERE, "golden", "bf16_bitfields.json")))["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["bits"])
def test_hand_fields(case):
    bits = int(case["bits"], 16)
    exp, sm = B.split(np.array([bits], dtype=np.uint16))
    assert (int(exp[0]), int(sm[0])) == (int(case["exp"], 16), int(case["sm"], 16))
    assert int(B.recombine(exp, sm)[0]) == bits


def test_fields_denote_the_value():
    """For every finite pattern the split fields, read by the IEEE definition, give the
    number torch decodes from the same bits (bf16 = upper half of a float32)."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    f32 = torch.from_numpy((bits << 16).astype(np.uint32).view(np.int32)).view(torch.float32).double().numpy()
    exp, sm = B.split(bits.astype(np.uint16))
    finite = exp != 0xFF
    rng = np.random.default_rng(0)
    for i in rng.choice(np.flatnonzero(finite), 4000, replace=False):
        assert B.value_of_fields(int(exp[i]), int(sm[i])) == f32[i]


def test_round_trip_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp, sm = B.split(bits)
    assert np.array_equal(B.recombine(exp, sm), bits)


def test_every_byte_pair_is_one_pattern():
    e, s = np.meshgrid(np.arange(256, dtype=np.uint8), np.arange(256, dtype=np.uint8), indexing="ij")
    bits = B.recombine(e.ravel(), s.ravel())
    assert np.unique(bits).size == 1 << 16
    e2, s2 = B.split(bits)
    assert np.array_equal(e2, e.ravel()) and np.array_equal(s2, s.ravel())


def test_entropy_closed_forms():
    assert B.exponent_entropy(np.full(100, 7, dtype=np.uint8)) == 0.0
    assert abs(B.exponent_entropy(np.arange(256, dtype=np.uint8)) - 8.0) < 1e-12
    assert abs(B.exponent_entropy(np.array([1, 1, 2, 3], dtype=np.uint8)) - 1.5) < 1e-12


def test_planted_mistake_is_caught():
    """A split that puts the sign in bit 0 of the SM byte fails the hand pins."""
    def bad_split(bits):
        b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
        return ((b >> 7) & 0xFF).astype(np.uint8), (((b & 0x7F) << 1) | (b >> 15)).astype(np.uint8)
    case = _golden()[1]   # -2.0
    exp, sm = bad_split(np.array([int(case["bits"], 16)], dtype=np.uint16))
    assert int(sm[0]) != int(case["sm"], 16)
