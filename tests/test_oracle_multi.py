"""Pins of the several-new-tokens oracle (chunked prefill / speculative decoding; CPU only).

New query i of a step that appended T tokens to a cache of S keys sits at position S - T + i
and sees keys 0 .. S - T + i: the causal mask aligned to the lower right ([W1D4] "第 1 周 ·
Day 4：KV Cache 与 MQA / GQA" §3.3, third case).  Pinned by:

- T = 1 is the single-token decode exactly;
- query i equals a single-token decode at length S - T + i + 1 (the definition, by slicing);
- chunked prefill through the cache equals the dense causal layer on the worked example
  ([W1D4] §3.5, first test, chunked form), which pins the mask's orientation;
- the append writes exactly slots [S - T, S).
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import synth


def _rand(shape, seed, dtype=np.float32):
    return np.ascontiguousarray(np.random.default_rng(seed).standard_normal(shape).astype(dtype))


def test_one_new_token_is_plain_decode():
    B, H_q, H_kv, T, D = 3, 8, 2, 12, 16
    Kc, Vc = _rand((B, H_kv, T, D), 1), _rand((B, H_kv, T, D), 2)
    q = _rand((B, H_q, 1, D), 3)
    lens = np.array([12, 5, 1], np.int32)
    got = oracle.decode_multi(q, Kc, Vc, lens)
    ref = oracle.decode_attn(np.ascontiguousarray(q[:, :, 0]), Kc, Vc, lens)
    assert np.array_equal(got[:, :, 0], ref)


@pytest.mark.parametrize("T_q", [2, 4, 7])
def test_query_i_is_single_token_decode_at_its_position(T_q):
    B, H_q, H_kv, T, D = 2, 4, 2, 20, 8
    Kc, Vc = _rand((B, H_kv, T, D), 4), _rand((B, H_kv, T, D), 5)
    q = _rand((B, H_q, T_q, D), 6)
    lens = np.array([20, T_q + 3], np.int32)
    got = oracle.decode_multi(q, Kc, Vc, lens)
    for i in range(T_q):
        li = (lens - T_q + i + 1).astype(np.int32)
        ref = oracle.decode_attn(np.ascontiguousarray(q[:, :, i]), Kc, Vc, li)
        assert np.array_equal(got[:, :, i], ref), i


@pytest.mark.parametrize("chunk", [1, 3, 5])
def test_chunked_prefill_through_the_cache_equals_the_dense_layer(chunk):
    B, hidden, H_q, H_kv, D, T = 1, 16, 4, 2, 4, 13
    Ws, x = synth.worked_example(7, hidden, H_q, H_kv, D, B, T)
    WQ, WK, WV, WO = Ws
    full, _, _ = oracle.layer_full(x.numpy(), *[w.numpy() for w in Ws], H_q, H_kv, D)
    q_all = (x @ WQ).view(B, T, H_q, D).transpose(1, 2).contiguous().numpy()   # [B,H_q,T,D]
    k_all = (x @ WK).view(B, T, H_kv, D).transpose(1, 2).contiguous().numpy()  # [B,H_kv,T,D]
    v_all = (x @ WV).view(B, T, H_kv, D).transpose(1, 2).contiguous().numpy()
    Kc = np.zeros((B, H_kv, T, D), np.float32)
    Vc = np.zeros_like(Kc)
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        lens = np.array([c1], np.int32)
        assert oracle.append_multi(Kc, Vc, np.ascontiguousarray(k_all[:, :, c0:c1]),
                                   np.ascontiguousarray(v_all[:, :, c0:c1]), lens) == 0
        o = oracle.decode_multi(np.ascontiguousarray(q_all[:, :, c0:c1]), Kc, Vc, lens)  # [B,H_q,n,D]
        y = torch.from_numpy(o).permute(0, 2, 1, 3).reshape(B, c1 - c0, H_q * D).float() @ WO
        np.testing.assert_allclose(y.numpy(), full[:, c0:c1], rtol=1e-4, atol=1e-5)
    assert np.array_equal(Kc, k_all) and np.array_equal(Vc, v_all)


def test_append_multi_writes_exactly_the_new_slots():
    B, H_kv, T, D, T_q = 3, 2, 10, 4, 3
    Kc, Vc = _rand((B, H_kv, T, D), 7), _rand((B, H_kv, T, D), 8)
    K0 = Kc.copy()
    kn, vn = _rand((B, H_kv, T_q, D), 9), _rand((B, H_kv, T_q, D), 10)
    lens = np.array([3, 10, 7], np.int32)
    assert oracle.append_multi(Kc, Vc, kn, vn, lens) == 0
    exp = K0.copy()
    for b in range(B):
        exp[b, :, lens[b] - T_q : lens[b]] = kn[b]
    assert np.array_equal(Kc, exp)
    assert oracle.append_multi(Kc, Vc, kn, vn, np.array([2, 11, 3], np.int32)) == 2  # L < T_q, L > T


def test_planted_upper_left_mask_is_caught():
    def fails(fn):
        try:
            fn()
        except AssertionError:
            return True
        return False
    with oracle.planted_fault(7):
        assert fails(test_one_new_token_is_plain_decode)
        assert fails(lambda: test_chunked_prefill_through_the_cache_equals_the_dense_layer(5))
