"""Pins of the float64 FP8 model (oracle/fp8.py) on the steps the model and
the kernel share by design: P rounded to e4m3 for the P V product while the
row sum takes the unrounded P, one e4m3 scale per head for V, and the lazy
rescale threshold of the online softmax.

The pages fix only the method -- FP8 with block quantisation and incoherent
processing ("FlashAttention 1, 2, and 3 Explained", section 4;
"FlashAttention and the Kernel Era", "The Breakthrough", the FP8 sentence) --
so each expected value here is derived by hand from the e4m3 number format
(1 sign, 4 exponent bits with bias 7, 3 mantissa bits: the quantum in the
binade [2^e, 2^(e+1)) is 2^(e-3), saturating at 448) and from the
online-softmax merge of "FlashAttention 1, 2, and 3 Explained", section 2
(two blocks joined by rescaling the first with e^(m_1 - m_2)).  The inputs are
built so that every score, block scale and V value is exact: the queries are
448 e_0 (block scale 1), each key block holds one row with 448 in channel 1
(block scale 1) and puts its score coefficient c_j in channel 0, and the
softmax scale is 1 / (448 log2 e), so the score of key j in log2 units is c_j.

Each pin is run once on the model as it stands and once on a copy with a
plausible mistake planted in one step (on the CPU, through monkeypatch): the
pin must fail on every planted mistake.
"""
import math

import numpy as np
import pytest

from oracle import fp8 as f8

SL2_SCALE = 1.0 / (448.0 * math.log2(math.e))  # softmax scale: score of key j = c_j (log2)


def scores_case(N, c, v_rows):
    """q [1, N, 1, 128] = 448 e_0; k with score coefficients c (dict key ->
    c_j, every other key -64, i.e. a weight of 2^-64 or less, which e4m3
    rounds to 0) and 448 in channel 1 of the first row of each 128-row block;
    v from v_rows (dict key -> (channel, value)), zero elsewhere."""
    q = np.zeros((1, N, 1, 128))
    q[0, :, 0, 0] = 448.0
    k = np.zeros((1, N, 1, 128))
    k[0, :, 0, 0] = -64.0
    for j, cj in c.items():
        k[0, j, 0, 0] = cj
    k[0, ::128, 0, 1] = 448.0
    v = np.zeros((1, N, 1, 128))
    for j, (ch, val) in v_rows.items():
        v[0, j, 0, ch] = val
    return q, k, v


# ---- pin 1: three keys, P rounded for P V, the row sum unrounded ----------

def pin_three_keys():
    # scores 0, -1.5, -2.25 (log2): P = 1, 2^-1.5 = 0.3535534, 2^-2.25 = 0.2102241.
    # e4m3: 2^-1.5 lies in [2^-2, 2^-1), quantum 2^-5: 11.31 quanta -> 11 -> 0.34375;
    #       2^-2.25 lies in [2^-3, 2^-2), quantum 2^-6: 13.45 quanta -> 13 -> 0.203125.
    # V rows 448 e_0, 224 e_1, 112 e_2 (head maximum 448: scale 1, all exact).
    q, k, v = scores_case(3, {0: 0.0, 1: -1.5, 2: -2.25}, {0: (0, 448.0), 1: (1, 224.0),
                                                             2: (2, 112.0)})
    o, lse = f8.attn_fwd_fp8(q, k, v, False, SL2_SCALE, rotate=False)
    l = 1.0 + 2.0 ** -1.5 + 2.0 ** -2.25          # the unrounded row sum
    want = np.zeros(128)
    want[:3] = [448.0, 0.34375 * 224.0, 0.203125 * 112.0]
    want /= l
    for i in range(3):
        np.testing.assert_allclose(o[0, i, 0], want, rtol=1e-12, atol=1e-12)
        assert abs(lse[0, 0, i] - math.log(l)) <= 1e-12


def test_pin_three_keys():
    pin_three_keys()


def test_pin_three_keys_fails_when_the_row_sum_takes_the_rounded_p(monkeypatch):
    monkeypatch.setattr(f8, "row_sum_terms", lambda p: f8.e4m3_round(p))
    with pytest.raises(AssertionError):
        pin_three_keys()


def test_pin_three_keys_fails_when_p_is_not_rounded(monkeypatch):
    monkeypatch.setattr(f8, "pv_operand", lambda p, quantize: p)
    with pytest.raises(AssertionError):
        pin_three_keys()


def test_pin_three_keys_fails_when_p_is_rounded_after_the_product(monkeypatch):
    # rounding (P V) instead of P: the product is summed unrounded
    orig = f8.pv_operand
    monkeypatch.setattr(f8, "pv_operand", lambda p, quantize: p * 1.0)
    monkeypatch.setattr(f8, "row_sum_terms", lambda p: orig(p, True))
    with pytest.raises(AssertionError):
        pin_three_keys()


# ---- pin 2: one e4m3 scale per head for V --------------------------------

def pin_v_head_scales(quantize_heads):
    v = np.zeros((1, 256, 2, 128))
    # head 0: maximum 896 (scale 2), and in rows 128.. a block whose own
    # maximum is 6.0.  0.0274 / 2 = 0.0137 lies in [2^-7, 2^-6), quantum 2^-10:
    # 14.03 quanta -> 14 -> 0.013671875, times 2 = 0.02734375.  (A scale for
    # the 128-row block alone, 6/448, would give 0.0274 / (6/448) = 2.0459
    # -> 2.0 -> 0.0267857.)
    v[0, 0, 0, 0] = 896.0
    v[0, 201, 0, 0] = 6.0
    v[0, 200, 0, 5] = 0.0274
    # head 1: maximum 1.0 (scale 1/448); 0.3 * 448 = 134.4 lies in [128, 256),
    # quantum 16: 8.4 quanta -> 8 -> 128, i.e. 128 / 448 = 2/7.  (One scale
    # for both heads, 2, would give 0.15 -> 0.15625 -> 0.3125.)
    v[0, 3, 1, 7] = 1.0
    v[0, 4, 1, 7] = 0.3
    y = quantize_heads(v)
    assert y[0, 0, 0, 0] == 896.0 and y[0, 201, 0, 0] == 6.0
    assert y[0, 200, 0, 5] == 0.02734375
    assert y[0, 3, 1, 7] == 1.0
    assert abs(y[0, 4, 1, 7] - 2.0 / 7.0) <= 1e-15


def quantize_heads_per_block(v, quantize=True):
    """A planted mistake: one scale per 128-row block of each head."""
    out = np.empty_like(v)
    for b in range(v.shape[0]):
        for h in range(v.shape[2]):
            for r0 in range(0, v.shape[1], 128):
                blk = v[b, r0:r0 + 128, h]
                m = float(np.abs(blk).max())
                s = m / f8.E4M3_MAX if m > 0 else 1.0
                out[b, r0:r0 + 128, h] = f8.e4m3_round(blk / s) * s
    return out


def quantize_heads_one_scale(v, quantize=True):
    """A planted mistake: one scale for the whole tensor."""
    m = float(np.abs(v).max())
    s = m / f8.E4M3_MAX if m > 0 else 1.0
    return f8.e4m3_round(v / s) * s


def test_pin_v_head_scales():
    pin_v_head_scales(f8.quantize_heads)


@pytest.mark.parametrize("mistake", [quantize_heads_per_block, quantize_heads_one_scale])
def test_pin_v_head_scales_fails_on_other_scalings(mistake):
    with pytest.raises(AssertionError):
        pin_v_head_scales(mistake)


# ---- pin 3: the lazy rescale, fired mid-row and not fired -----------------

def pin_threshold_fires():
    # block 0: key 0 at score 0, the rest 2^-64 below (rounded to 0 for P V).
    # block 1: keys 128, 130 at 10 and key 129 at 9: the block maximum exceeds
    # the reference (0) by more than 8, so the reference moves to 10 and block
    # 0's sum and output are scaled by 2^-10 (the two-block merge).  Then
    # P = 1, 0.5, 1 (exact in e4m3), l = 2^-10 + 2.5.  V: 448 e_0 (key 0),
    # 256 e_1, 64 e_2 (keys 128, 129), 0.0274 e_3 (key 130), head scale 1:
    # 0.0274 lies in [2^-6, 2^-5), quantum 2^-9: 14.03 -> 14 -> 14 * 2^-9.
    q, k, v = scores_case(256, {0: 0.0, 128: 10.0, 129: 9.0, 130: 10.0},
                          {0: (0, 448.0), 128: (1, 256.0), 129: (2, 64.0), 130: (3, 0.0274)})
    o, lse = f8.attn_fwd_fp8(q, k, v, False, SL2_SCALE, rotate=False)
    l = 2.0 ** -10 + 2.5
    want = np.zeros(128)
    want[:4] = [2.0 ** -10 * 448.0, 256.0, 32.0, 14 * 2.0 ** -9]
    want /= l
    for i in (0, 100, 255):
        np.testing.assert_allclose(o[0, i, 0], want, rtol=1e-12, atol=1e-15)
        assert abs(lse[0, 0, i] - (10.0 + math.log2(l)) * math.log(2.0)) <= 1e-12


def pin_threshold_holds():
    # block 1's maximum, 5.5, is within 8 of the reference 0, which stays:
    # P of key 128 is 2^5.5 = 45.2548, in [32, 64), quantum 4: 11.31 -> 11 -> 44
    # for P V, while l adds the unrounded 45.2548.  (Moving the reference to
    # 5.5 would round P = 1 exactly and give 256 * 45.2548 in channel 1.)
    q, k, v = scores_case(256, {0: 0.0, 128: 5.5}, {0: (0, 448.0), 128: (1, 256.0)})
    o, lse = f8.attn_fwd_fp8(q, k, v, False, SL2_SCALE, rotate=False)
    l = 1.0 + 2.0 ** 5.5
    want = np.zeros(128)
    want[:2] = [448.0, 44.0 * 256.0]
    want /= l
    np.testing.assert_allclose(o[0, 0, 0], want, rtol=1e-12, atol=1e-15)
    assert abs(lse[0, 0, 0] - math.log(l)) <= 1e-12


def test_pin_threshold_fires():
    pin_threshold_fires()


def test_pin_threshold_holds():
    pin_threshold_holds()


def test_pin_threshold_holds_fails_with_an_eager_rescale(monkeypatch):
    # threshold 0: the reference follows every new maximum
    monkeypatch.setattr(f8, "LAZY_THRESHOLD", 0.0)
    with pytest.raises(AssertionError):
        pin_threshold_holds()


def test_pin_threshold_fires_fails_with_a_larger_threshold(monkeypatch):
    # threshold 16: the reference stays at 0 and P = 2^10 saturates at 448
    monkeypatch.setattr(f8, "LAZY_THRESHOLD", 16.0)
    with pytest.raises(AssertionError):
        pin_threshold_fires()


def test_pin_threshold_fires_fails_with_per_block_v_scales(monkeypatch):
    # keys 128..130 share a block whose own maximum is 256: a block scale
    # would round 0.0274 differently (0.0274 / (256/448) = 0.04795 -> 0.046875)
    monkeypatch.setattr(f8, "quantize_heads", quantize_heads_per_block)
    with pytest.raises(AssertionError):
        pin_threshold_fires()
