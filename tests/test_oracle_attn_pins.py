"""Pins of the decode-attention oracle (oracle/attn_oracle.c) to facts that do
not come from the oracle itself: closed forms of the rotary embedding, and
special weight choices under which the attention step reduces to something
computable by hand (a single visible key, uniform attention, the sliding
window, grouped-query sharing, invariance to a shift of every position).

Weights built here are canonical 4-bit tensors with scale 1 and bias 0, so
a code c is exactly the value c: selection matrices pick input columns."""
import math

import numpy as np
import pytest

import oracle
import synth


class Shape:
    d_model, n_heads, n_kv_heads, head_dim, group = 128, 2, 1, 64, 64


ONE = np.uint16(0x3C00)  # fp16 1.0


def qt_from_codes(codes):
    """Canonical 4-bit tensor with value = code (scale 1, bias 0)."""
    codes = np.asarray(codes, np.uint8)
    rows, cols = codes.shape
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s = np.full((rows, cols // 64), ONE, np.uint16)
    b = np.zeros((rows, cols // 64), np.uint16)
    return (q, s, b)


def select(rows, cols, offset=0):
    c = np.zeros((rows, cols), np.uint8)
    for r in range(rows):
        c[r, (r + offset) % cols] = 1
    return c


def tokens(n, D, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, D)).astype(np.float32)
    u = x.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)  # bf16 bits, nearest even


def bf16_to_f64(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def unit_rms(v):
    return v / math.sqrt(np.mean(v * v) + 1e-6)


def f16(v):
    return np.asarray(v, np.float64).astype(np.float16).astype(np.float64)


# ------------------------------------------------------------------ rotary

def test_rope_closed_forms():
    # position 0 is the identity
    v = np.random.default_rng(0).standard_normal(64)
    assert np.array_equal(oracle.rope(v, 0, 10000.0), v)
    # d = 2, position 1: the pair rotates by exactly 1 radian
    r = oracle.rope(np.array([1.0, 0.0]), 1, 10000.0)
    assert np.allclose(r, [math.cos(1.0), math.sin(1.0)], rtol=0, atol=1e-15)
    # pair i of d = 4 at position 3 rotates by 3 * theta^(-2i/4)
    r = oracle.rope(np.array([1.0, 1.0, 0.0, 0.0]), 3, 100.0)
    assert np.allclose(r, [math.cos(3.0), math.cos(0.3), math.sin(3.0), math.sin(0.3)], atol=1e-15)


def test_rope_is_a_rotation_that_depends_on_relative_position():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n in [(5, 2), (100, 37), (4096, 4000)]:
        a = oracle.rope(q, m, 1e6) @ oracle.rope(k, n, 1e6)
        b = oracle.rope(q, m - n, 1e6) @ k
        assert abs(a - b) <= 1e-9 * (1 + abs(a))
        assert abs(np.linalg.norm(oracle.rope(q, m, 1e6)) - np.linalg.norm(q)) < 1e-12


def test_head_rms_is_unit_gain_and_scale_free():
    v = np.random.default_rng(2).standard_normal(256) * 7.0
    u = oracle.head_rms(v)
    assert abs(np.mean(u * u) - 1.0) < 1e-6
    assert np.allclose(oracle.head_rms(v * 1000.0), u, rtol=1e-7)   # eps is not scaled
    assert np.all(oracle.head_rms(np.zeros(8)) == 0)


# ------------------------------------------------------------- attention

def attn_state(wq_codes, cap, window, theta=10000.0):
    sh = Shape
    w = {"wq": qt_from_codes(wq_codes), "wk": qt_from_codes(select(64, 128, 3)),
         "wv": qt_from_codes(select(64, 128)), "wo": qt_from_codes(select(128, 128))}
    return oracle.AttnState(sh, w, cap, window, theta)


def v_hat(x_bits):
    """The value vector a token stores under the selection weights: the first
    64 values of its pre-normed input, RMS-normalised, in fp16."""
    u = unit_rms(bf16_to_f64(x_bits))
    return f16(unit_rms(u[:64]))


def test_single_visible_key_returns_its_value_whatever_the_query():
    xs = tokens(1, 128, 3)
    rng = np.random.default_rng(4)
    for wq in (np.zeros((128, 128), np.uint8), rng.integers(0, 16, (128, 128)).astype(np.uint8)):
        st = attn_state(wq, cap=16, window=0)
        y = st.step(xs[0], 0)
        # both query heads read the one key/value head; Wo is the identity
        assert np.array_equal(y[:64], v_hat(xs[0])) and np.array_equal(y[64:], v_hat(xs[0]))


def test_zero_query_averages_the_window_and_heads_share_their_kv_head():
    """Wq = 0 makes every score 0: the output is the plain mean of the stored
    values of the visible positions, the last `window` ones in a ring of
    that size, or all of them in a linear cache."""
    xs = tokens(7, 128, 5)
    ring = attn_state(np.zeros((128, 128), np.uint8), cap=3, window=3)
    lin = attn_state(np.zeros((128, 128), np.uint8), cap=16, window=0)
    for p in range(7):
        yr = ring.step(xs[p], p)
        yl = lin.step(xs[p], p)
        want_r = np.mean([v_hat(xs[j]) for j in range(max(0, p - 2), p + 1)], axis=0)
        want_l = np.mean([v_hat(xs[j]) for j in range(p + 1)], axis=0)
        assert np.allclose(yr[:64], want_r, rtol=0, atol=1e-12), p
        assert np.allclose(yl[:64], want_l, rtol=0, atol=1e-12), p
        assert np.array_equal(yr[:64], yr[64:]) and np.array_equal(yl[:64], yl[64:])


def test_shifting_every_position_changes_nothing_but_rounding():
    """With RoPE only relative positions matter: the same six tokens attended
    at positions 0..5 and at 9..14, through a six-token window (so the second
    run sees exactly its own tokens, in ring slots 3..2), give the same
    output; the cached keys are rotated, then rounded to fp16, so the two
    agree to fp16 precision."""
    sh = synth.TINY_ATTN
    w = synth.make_attn_layer(sh, "tiny", 0)
    xs = tokens(6, sh.d_model, 6)
    a = oracle.AttnState(sh, w, 6, 6, 10000.0)
    b = oracle.AttnState(sh, w, 6, 6, 10000.0)
    for p in range(6):
        ya = a.step(xs[p], p)
        yb = b.step(xs[p], p + 9)
    assert np.abs(ya - yb).max() <= 3e-3 * np.sqrt(np.mean(ya ** 2))


def test_bad_arguments_are_refused():
    st = attn_state(np.zeros((128, 128), np.uint8), cap=4, window=0)
    with pytest.raises(ValueError):
        st.step(tokens(1, 128, 7)[0], 4)          # beyond a linear cache


def test_grouped_query_heads_read_their_own_kv_head():
    """Hq = 4 over Hkv = 2: query heads 0, 1 read kv head 0 and heads 2, 3 read
    kv head 1 (zero queries, so each is the mean of its kv head's values)."""
    class Sh:
        d_model, n_heads, n_kv_heads, head_dim, group = 256, 4, 2, 64, 64

    w = {"wq": qt_from_codes(np.zeros((256, 256), np.uint8)),
         "wk": qt_from_codes(select(128, 256, 5)), "wv": qt_from_codes(select(128, 256)),
         "wo": qt_from_codes(select(256, 256))}
    st = oracle.AttnState(Sh, w, 8, 0, 10000.0)
    xs = tokens(3, 256, 8)
    for p in range(3):
        y = st.step(xs[p], p)

    def vh(x, lo):
        u = unit_rms(bf16_to_f64(x))
        return f16(unit_rms(u[lo:lo + 64]))

    want0 = np.mean([vh(xs[j], 0) for j in range(3)], axis=0)
    want1 = np.mean([vh(xs[j], 64) for j in range(3)], axis=0)
    for h, want in ((0, want0), (1, want0), (2, want1), (3, want1)):
        assert np.allclose(y[64 * h:64 * h + 64], want, rtol=0, atol=1e-12), h


def test_score_scale_is_one_over_sqrt_head_dim():
    """Queries equal to keys (same selection of the input), a first token
    whose key is exactly zero (score 0) and a second whose key equals its own
    query: the second score is |k|^2 / sqrt(d) = d / sqrt(d) = 8 up to the fp16
    rounding of the stored key, so the weights are (1, e^8) / (1 + e^8)."""
    w = {"wq": qt_from_codes(select(128, 128) * 0 + np.vstack([select(64, 128)] * 2)),
         "wk": qt_from_codes(select(64, 128)), "wv": qt_from_codes(select(64, 128, 64)),
         "wo": qt_from_codes(select(128, 128))}
    st = oracle.AttnState(Shape, w, 8, 0, 10000.0)
    xs = tokens(2, 128, 9)
    xs[0, :64] = 0                                    # key of token 0 is exactly zero
    st.step(xs[0], 0)
    y = st.step(xs[1], 1)

    def vh(x):
        u = unit_rms(bf16_to_f64(x))
        return f16(unit_rms(u[64:128]))

    w1 = 1.0 / (1.0 + math.exp(-8.0))
    want = (1 - w1) * vh(xs[0]) + w1 * vh(xs[1])
    err = np.abs(y[:64] - want).max()
    assert err <= 2e-3 * np.abs(want).max(), err
    assert np.array_equal(y[:64], y[64:])
