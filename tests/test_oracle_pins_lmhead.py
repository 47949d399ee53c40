"""Pins of the oracle's storage decoding, lm-head and argmax-margin helpers.

These helpers decide what every GPU parity test compares: `bf16_to_f64`
decodes the embedding and lm-head tables, `lmhead_logits` / `lmhead_argmax`
produce the draft tokens, and `top2_margin` picks which draft positions are
compared at all (only where the oracle's top-2 logit gap exceeds 1e-2).  Each
pin uses values fixed independently of the oracle: bit patterns decoded by
hand from the bfloat16 format (1 sign bit, 8 exponent bits with bias 127, 7
fraction bits), logits worked out by hand from small integer tables, and gaps
read off hand-written rows.  Every pin has a negative control: a plausible
mistake planted in the oracle (on the CPU) that the same check rejects.
"""
import numpy as np
import pytest

from oracle import dflash_oracle as O

# (bits, value) pairs decoded by hand from the bfloat16 layout
BF16_CASES = [
    (0x3F80, 1.0),                          # sign 0, exponent 127, fraction 0
    (0xC020, -2.5),                         # sign 1, exponent 128, fraction 0x20 = 0.25 -> -(1.25 * 2)
    (0x4049, 3.140625),                     # exponent 128, fraction 0x49 / 128 = 0.5703125 -> 1.5703125 * 2
    (0x0000, 0.0),
    (0x8000, -0.0),
    (0x0001, 2.0 ** -133),                  # smallest subnormal: 1/128 * 2^-126
    (0x0080, 2.0 ** -126),                  # smallest normal
    (0x007F, 127.0 / 128.0 * 2.0 ** -126),  # largest subnormal
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),  # largest finite
    (0x7F80, np.inf),
    (0xFF80, -np.inf),
    (0x3C00, 2.0 ** -7),                    # exponent 120
]


def _bf16_pin(decode) -> bool:
    bits = np.array([b for b, _ in BF16_CASES], np.uint16)
    want = np.array([v for _, v in BF16_CASES], np.float64)
    got = np.asarray(decode(bits), np.float64)
    if got.shape != want.shape or not np.array_equal(got, want):
        return False
    # the sign of zero is part of the pattern
    return bool(np.signbit(got[4])) and not bool(np.signbit(got[3]))


def test_bf16_decoding_matches_hand_decoded_patterns():
    assert _bf16_pin(O.bf16_to_f64)
    # 2-D input keeps its shape
    two = O.bf16_to_f64(np.array([[0x3F80, 0xC020], [0x4049, 0x0001]], np.uint16))
    assert two.shape == (2, 2) and two[0, 1] == -2.5


def test_bf16_decoding_negative_controls():
    # read as fp16 bits
    assert not _bf16_pin(lambda b: np.asarray(b, np.uint16).view(np.float16).astype(np.float64))
    # shifted into the wrong half of the fp32 word
    assert not _bf16_pin(lambda b: np.asarray(b, np.uint16).astype(np.uint32).view(np.float32).astype(np.float64))
    # rounded through fp16 on the way (loses the range of bf16)
    with np.errstate(over="ignore"):
        assert not _bf16_pin(lambda b: O.bf16_to_f64(b).astype(np.float16).astype(np.float64))


# --------------------------------------------------------------- margins ----
MARGIN_ROWS = [
    ([1.0, 3.0, 2.5, -1.0], 0.5),
    ([4.0, 1.0, 4.0], 0.0),             # tied maximum: no margin
    ([-3.0, -1.0, -2.0], 1.0),          # all negative: top -1, second -2
    ([-5.0, -5.5], 0.5),
    ([7.0, 7.0, 7.0, 2.0], 0.0),
    ([0.25, -10.0, 0.125, 0.0], 0.125),
]


def _margin_pin(fn) -> bool:
    for row, gap in MARGIN_ROWS:
        if float(fn(np.array(row, np.float64))) != gap:
            return False
    # batched over leading axes, row by row
    batch = np.array([MARGIN_ROWS[0][0], [2.0, 9.0, 8.0, 1.0]], np.float64)
    return np.array_equal(np.asarray(fn(batch)), np.array([0.5, 1.0]))


def test_top2_margin_hand_worked_rows():
    assert _margin_pin(O.top2_margin)


def test_top2_margin_negative_controls():
    # top-1 minus minimum
    assert not _margin_pin(lambda x: x.max(axis=-1) - x.min(axis=-1))
    # gap between the two largest distinct values (a tie would not count)
    def distinct(x):
        x = np.atleast_2d(x)
        out = np.array([np.sort(np.unique(r))[-1] - np.sort(np.unique(r))[-2] for r in x])
        return out if out.size > 1 else out[0]
    assert not _margin_pin(distinct)
    # gap of absolute values (wrong on negative rows)
    assert not _margin_pin(lambda x: O.top2_margin(np.abs(x)))


# --------------------------------------------------------------- lm-head ----
def _table(V: int, H: int) -> np.ndarray:
    """bf16 bits of W[v][j] = (v - 4) / 2 + j, small integers and halves
    (exact in bf16): hand-encoded as 1.f * 2^e."""
    def enc(x: float) -> int:
        if x == 0.0:
            return 0x0000
        s = 0x8000 if x < 0 else 0
        m, e = np.frexp(abs(x))          # abs(x) = m 2^e, m in [0.5, 1)
        frac = int(round((m * 2 - 1) * 128))
        assert (m * 2 - 1) * 128 == frac  # exactly representable
        return s | ((int(e) - 1 + 127) << 7) | frac
    W = np.zeros((V, H), np.uint16)
    for v in range(V):
        for j in range(H):
            W[v, j] = enc((v - 4) / 2 + j)
    return W


def _lm_pin(logits_fn, chunk: int) -> bool:
    V, H = 2 * chunk + 3, 3
    W = _table(V, H)
    # one-hot rows pick a column of W; a two-term row mixes two
    h = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 1.0], [2.0, 0.0, -1.0]], np.float64)
    lg = logits_fn(h, W, chunk)
    v = np.arange(V, dtype=np.float64)
    want = np.stack([(v - 4) / 2, (v - 4) / 2 + 2, 2 * ((v - 4) / 2) - ((v - 4) / 2 + 2)])
    return lg.shape == want.shape and np.array_equal(lg, want)


@pytest.mark.parametrize("chunk", [1, 2, 4, 5])
def test_lmhead_logits_hand_built_table(chunk):
    # V spans chunk boundaries (2 chunk + 3 rows): every row must be computed once
    assert _lm_pin(lambda h, W, c: O.lmhead_logits(h, W, chunk=c), chunk)


def test_lmhead_logits_negative_controls():
    def skip_last_of_chunk(h, W, chunk):
        lg = O.lmhead_logits(h, W, chunk=chunk)
        lg[:, chunk - 1::chunk] = 0.0
        return lg

    def reversed_vocab(h, W, chunk):  # vocabulary rows indexed from the wrong end
        return np.asarray(h, np.float64) @ O.bf16_to_f64(W[::-1]).T

    assert not _lm_pin(skip_last_of_chunk, 4)
    assert not _lm_pin(reversed_vocab, 4)


def test_lmhead_argmax_hand_worked():
    # vocabulary of 9, hidden 2; W rows chosen so row 0 of h = e0 peaks at a
    # tie between v = 3 and v = 7 (lowest wins), row 1 = -e1 peaks at v = 0
    one, half, two, neg1, neg2 = 0x3F80, 0x3F00, 0x4000, 0xBF80, 0xC000
    W = np.array([
        [half, neg2],   # v0:  0.5, -2
        [neg1, one],    # v1: -1,   1
        [0x0000, two],  # v2:  0,   2
        [two, 0x0000],  # v3:  2,   0
        [one, neg1],    # v4:  1,  -1
        [half, one],    # v5:  0.5, 1
        [neg2, two],    # v6: -2,   2
        [two, half],    # v7:  2,   0.5
        [one, 0x0000],  # v8:  1,   0
    ], np.uint16)
    h = np.array([[one, 0x0000], [0x0000, neg1]], np.uint16)
    idx, mx, margin, lg = O.lmhead_argmax(h, W)
    assert list(idx) == [3, 0]
    assert list(mx) == [2.0, 2.0]
    # row 0: 2 (v3, v7) then 1: tie -> gap 0; row 1: 2 (v0) then 1 (v4): gap 1
    assert list(margin) == [0.0, 1.0]
    assert np.array_equal(lg[1], [2.0, -1.0, -2.0, 0.0, 1.0, -1.0, -2.0, -0.5, 0.0])


def test_lmhead_argmax_negative_control(monkeypatch):
    # an argmax that keeps the LAST of tied maxima changes the draft token
    W = np.array([[0x4000], [0x3F80], [0x4000]], np.uint16)
    h = np.array([[0x3F80]], np.uint16)
    assert O.lmhead_argmax(h, W)[0][0] == 0
    monkeypatch.setattr(O, "argmax_lowest", lambda x: x.shape[-1] - 1 - np.argmax(x[..., ::-1], axis=-1))
    assert O.lmhead_argmax(h, W)[0][0] == 2
