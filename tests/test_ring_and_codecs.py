"""Pins of the cursor model and the read-copy codecs.

RingModel is checked exhaustively against a naive model that keeps the
buffered records in an explicit list and a slot array; the codecs against
the OCP bit-field definitions, hand-listed rounding cases and torch's own
float8_e4m3fn conversion.
"""

import itertools

import numpy as np
import pytest
import torch

from oracle import codecs
from oracle.ring import RingModel


class NaiveRing:
    """Explicit record list plus slot array: a record is written to the next
    free slot after the last committed one; a fold empties the list."""

    def __init__(self, L, C):
        self.L, self.C = L, C
        self.slots = [None] * C
        self.records = []          # ids of committed records since the last fold
        self.next_slot = 0         # slot of the first record after the last fold
        self.drafts = []
        self.uid = 0

    def _write(self, pos):
        rid = self.uid
        self.uid += 1
        self.slots[(self.next_slot + pos) % self.C] = rid
        return rid

    def _fold(self):
        self.next_slot = (self.next_slot + len(self.records)) % self.C
        self.records = []

    def decode(self):
        self.records.append(self._write(len(self.records)))
        if len(self.records) == self.L:
            self._fold()
            return 1
        return 0

    def verify(self, T):
        self.drafts = [self._write(len(self.records) + i) for i in range(T)]

    def commit(self, n):
        self.records += self.drafts[:n]
        self.drafts = []
        if len(self.records) >= self.L:
            self._fold()
            return 1
        return 0

    def flush(self):
        self._fold()


def _check_same(m, nv):
    assert m.count == len(nv.records)
    assert m.head == nv.next_slot
    for j, rid in enumerate(nv.records):
        assert nv.slots[m.slot(j)] == rid


@pytest.mark.parametrize("L,T", [(1, 1), (2, 1), (3, 2), (4, 3), (4, 2)])
def test_ring_exhaustive_speculative(L, T):
    """All sequences of accepted counts over 6 verify/commit rounds."""
    C = L + T
    for seq in itertools.product(range(T + 1), repeat=6):
        m, nv = RingModel(L, C), NaiveRing(L, C)
        for n in seq:
            m.verify(T)
            nv.verify(T)
            assert m.commit(n) == nv.commit(n)
            _check_same(m, nv)
            assert m.count < L


@pytest.mark.parametrize("L", [1, 2, 4, 16])
def test_ring_exhaustive_mixed_calls(L):
    """Every interleaving of decode / verify+commit / flush of length 8 (T = 2)."""
    T = 2
    C = L + T
    ops = ["decode", "flush"] + [("spec", n) for n in range(T + 1)]
    for seq in itertools.product(ops, repeat=5 if L > 4 else 6):
        m, nv = RingModel(L, C), NaiveRing(L, C)
        for op in seq:
            if op == "decode":
                assert m.decode() == nv.decode()
            elif op == "flush":
                m.flush()
                nv.flush()
            else:
                m.verify(T)
                nv.verify(T)
                assert m.commit(op[1]) == nv.commit(op[1])
            _check_same(m, nv)


def test_ring_rules():
    m = RingModel(4, 6)
    m.verify(2)
    with pytest.raises(RuntimeError):
        m.decode()
    with pytest.raises(RuntimeError):
        m.verify(1)
    with pytest.raises(ValueError):
        m.commit(3)
    m.commit(2)
    with pytest.raises(ValueError):
        m.verify(5)


# --- codecs ----------------------------------------------------------------------

def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = codecs.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_landmarks():
    """Published E4M3 landmarks: max 448, min normal 2^-6, min subnormal 2^-9."""
    assert codecs.e4m3_decode(0x7E) == 448.0
    assert codecs.e4m3_decode(0x08) == 2.0 ** -6
    assert codecs.e4m3_decode(0x01) == 2.0 ** -9
    assert codecs.e4m3_decode(0x38) == 1.0
    assert codecs.e4m3_decode(0xB8) == -1.0


def test_e4m3_encode_rne_cases():
    cases = {
        1.0625: 0x38,        # halfway 1 and 1.125 -> even mantissa (1.0)
        1.1875: 0x3A,        # halfway 1.125 and 1.25 -> 1.25 (even)
        2.0 ** -10: 0x00,    # halfway 0 and 2^-9 -> 0
        3 * 2.0 ** -10: 0x02,  # halfway 2^-9 and 2^-8 -> 2^-8 (even code)
        1000.0: 0x7E,        # saturates to 448
        -1e30: 0xFE,
        464.0: 0x7E,
        -0.0: 0x80,
    }
    for x, c in cases.items():
        assert int(codecs.e4m3_encode(np.float64(x))) == c, (x, c)


def test_e4m3_encode_matches_torch_cast():
    r = np.random.default_rng(7)
    x = np.concatenate([r.standard_normal(200000) * s for s in (1e-3, 1e-1, 1.0, 30.0, 200.0)])
    x = x[np.abs(x) <= 448.0].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codecs.e4m3_encode(x), ref)


def test_e4m3_roundtrip_all_finite():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = codecs.e4m3_encode(codecs.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def test_e2m1_table_and_rounding():
    vals = codecs.e2m1_decode(np.arange(16))
    assert vals.tolist() == [0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 5.5: 7, 7.0: 7,
             100.0: 7, -0.25: 8, -2.6: 13, 0.3: 1}
    for x, c in cases.items():
        assert int(codecs.e2m1_encode(np.float64(x))) == c, (x, c)


def test_fp8_rows_error_bound():
    r = np.random.default_rng(3)
    S = (0.05 * r.standard_normal((3, 16, 32))).astype(np.float32)
    S[0, 0] = 0.0
    codes, sc = codecs.fp8_rows_quantize(S)
    assert sc[0, 0] == 0 and not codes[0, 0].any()
    Rq = codecs.fp8_rows_dequantize(codes, sc)
    amax = np.abs(S).max(axis=-1, keepdims=True)
    # relative half-ulp of a 3-bit mantissa, plus the subnormal floor
    bound = np.abs(S) * 2.0 ** -4 + (amax / 448.0) * 2.0 ** -10 + 1e-12
    assert np.all(np.abs(Rq - S) <= bound * 1.0001)
    # the row maximum is represented (scaled to 448) up to float32 rounding
    i = np.unravel_index(np.argmax(np.abs(S[1, 2])), S[1, 2].shape)
    assert abs(abs(Rq[1, 2][i]) - amax[1, 2, 0]) <= 1e-6 * amax[1, 2, 0]


def test_nvfp4_structure_and_error_bound():
    r = np.random.default_rng(4)
    S = (0.1 * r.standard_normal((2, 8, 64))).astype(np.float32)
    packed, bs, s = codecs.nvfp4_quantize(S)
    assert packed.shape == (2, 8, 32) and bs.shape == (2, 8, 4) and s.shape == (2,)
    assert np.all(codecs.e4m3_decode(bs) <= 448.0)
    Rq = codecs.nvfp4_dequantize(packed, bs, s)
    blk = np.abs(S).reshape(2, 8, 4, 16).max(axis=-1)
    dscale = codecs.e4m3_decode(bs) * s[:, None, None]
    # each element within half an e2m1 step (at most 1 unit of the block scale)
    # of its value, plus the block-scale rounding of the block maximum
    err = np.abs(Rq - S).reshape(2, 8, 4, 16)
    assert np.all(err <= (dscale * 1.0 + blk * 2.0 ** -3)[..., None] * 1.0001 + 1e-9)
    # packing: element 2i in the low nibble
    codes_lo = packed & 0xF
    ref = codecs.e2m1_encode((S[..., 0::2] / np.repeat(dscale, 8, axis=-1).astype(np.float32)).astype(np.float32))
    assert np.array_equal(codes_lo, ref)
    # all-zero matrix
    z = np.zeros((1, 4, 32), np.float32)
    p0, b0, s0 = codecs.nvfp4_quantize(z)
    assert not p0.any() and not b0.any() and s0[0] == 0
