"""Pins of the sliding-window / rolling-cache oracle (CPU only).

With a window of W tokens the newest query attends to the W most recent positions and the
cache keeps W slots, position p in slot p mod W ([W1D4] "第 1 周 · Day 4：KV Cache 与 MQA / GQA"
§2.7 and §1.6; [M11] "11.7 KV Cache：形状、显存与带宽" §8).  Pinned against the plain decode
oracle (itself pinned in test_oracle_pins.py) on explicitly sliced histories, and against the
rolling cache fed one token at a time:

- window >= length: identical to plain decode;
- window W: identical to plain decode over the sliced history [L-W, L);
- window 1: the output is the newest value row;
- a rolling cache fed token by token gives exactly the window result over the full history;
- the append writes slot (L-1) mod W and nothing else.
"""
import numpy as np
import pytest

import oracle


def _rand(shape, seed, dtype=np.float32):
    return np.ascontiguousarray(np.random.default_rng(seed).standard_normal(shape).astype(dtype))


def test_window_at_least_length_is_plain_decode():
    B, H_q, H_kv, T, D = 3, 8, 2, 20, 16
    Kc, Vc, q = _rand((B, H_kv, T, D), 1), _rand((B, H_kv, T, D), 2), _rand((B, H_q, D), 3)
    lens = np.array([20, 7, 1], np.int32)
    ref = oracle.decode_attn(q, Kc, Vc, lens)
    for W in (20, 21, 1000):
        assert np.array_equal(oracle.window_decode_attn(q, Kc, Vc, lens, W), ref)


@pytest.mark.parametrize("W", [1, 3, 8])
def test_window_equals_decode_over_the_sliced_history(W):
    B, H_q, H_kv, T, D = 3, 4, 2, 16, 8
    Kc, Vc, q = _rand((B, H_kv, T, D), 4), _rand((B, H_kv, T, D), 5), _rand((B, H_q, D), 6)
    lens = np.array([16, 9, 2], np.int32)
    got = oracle.window_decode_attn(q, Kc, Vc, lens, W)
    for b in range(B):
        L = int(lens[b])
        t0 = max(0, L - W)
        Ks = np.ascontiguousarray(Kc[b : b + 1, :, t0:L])
        Vs = np.ascontiguousarray(Vc[b : b + 1, :, t0:L])
        ref = oracle.decode_attn(np.ascontiguousarray(q[b : b + 1]), Ks, Vs, np.array([L - t0], np.int32))
        assert np.array_equal(got[b : b + 1], ref)


def test_window_one_returns_the_newest_value_row():
    B, H_q, H_kv, T, D = 2, 6, 3, 10, 4
    Kc, Vc, q = _rand((B, H_kv, T, D), 7), _rand((B, H_kv, T, D), 8), _rand((B, H_q, D), 9)
    lens = np.array([10, 4], np.int32)
    got = oracle.window_decode_attn(q, Kc, Vc, lens, 1)
    for b in range(B):
        for j in range(H_q):
            assert np.array_equal(got[b, j], Vc[b, j // 2, lens[b] - 1].astype(np.float64))


@pytest.mark.parametrize("W", [1, 4, 7])
def test_rolling_cache_fed_token_by_token_equals_the_window(W):
    B, H_q, H_kv, D, T = 2, 4, 2, 8, 19
    K, V = _rand((B, H_kv, T, D), 10), _rand((B, H_kv, T, D), 11)
    Kr = np.zeros((B, H_kv, W, D), np.float32)
    Vr = np.zeros_like(Kr)
    for step in range(T):
        # sequence 1 stays at length 1 for its first steps (its token 0 rewritten in place)
        lens = np.array([step + 1, max(1, step - 3)], np.int32)
        kn = np.ascontiguousarray(K[np.arange(B), :, lens - 1])
        vn = np.ascontiguousarray(V[np.arange(B), :, lens - 1])
        assert oracle.rolling_append(Kr, Vr, kn, vn, lens) == 0
        q = _rand((B, H_q, D), 100 + step)
        got = oracle.rolling_decode_attn(q, Kr, Vr, lens)
        ref = oracle.window_decode_attn(q, K, V, lens, W)
        assert np.array_equal(got, ref), step


def test_rolling_append_writes_one_slot():
    B, H_kv, W, D = 3, 2, 5, 4
    Kr, Vr = _rand((B, H_kv, W, D), 12), _rand((B, H_kv, W, D), 13)
    K0 = Kr.copy()
    kn, vn = _rand((B, H_kv, D), 14), _rand((B, H_kv, D), 15)
    lens = np.array([1, 5, 13], np.int32)
    assert oracle.rolling_append(Kr, Vr, kn, vn, lens) == 0
    exp = K0.copy()
    for b in range(B):
        exp[b, :, (lens[b] - 1) % W] = kn[b]
    assert np.array_equal(Kr, exp)
    bad = np.array([0, 2, 3], np.int32)
    assert oracle.rolling_append(Kr, Vr, kn, vn, bad) == 1


def test_planted_wide_window_is_caught():
    def fails(fn):
        try:
            fn()
        except AssertionError:
            return True
        return False
    with oracle.planted_fault(6):
        assert fails(lambda: test_window_equals_decode_over_the_sliced_history(3))
        assert fails(test_window_one_returns_the_newest_value_row)
