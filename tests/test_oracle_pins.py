"""Pins for the CPU oracle: what the pages and the mathematics fix, independent of the oracle.

Each planted mistake (oracle.planted_fault) must make at least one of these fail; the
last tests check exactly that.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, dtype=np.float32):
    return np.ascontiguousarray(np.random.default_rng(seed).standard_normal(shape).astype(dtype))


def _f64(a):
    return oracle.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


# ---------------------------------------------------------------------------- capacity
def _golden_capacity():
    rows = []
    for line in open(os.path.join(GOLDEN, "capacity.txt"), encoding="utf-8"):
        if not line.strip() or line.startswith("#"):
            continue
        name, dims, expected, kind, src = [c.strip() for c in line.split("|")]
        rows.append((name, [int(x) for x in dims.split()], float(expected), kind, src))
    return rows


@pytest.mark.parametrize("name,dims,expected,kind,src", _golden_capacity())
def test_capacity_closed_forms(name, dims, expected, kind, src):
    L, B, H_kv, D, T, s = dims
    got = oracle.kv_bytes(L, B, H_kv, D, T, s)
    if kind == "exact":
        assert got == int(expected), (name, src)
    elif kind == "GiB~":
        assert round(got / 2**30) == int(expected), (name, got / 2**30, src)
    elif kind == "MiB~":
        assert f"{got / 2**20:.3f}" == f"{expected:.3f}", (name, got / 2**20, src)
    else:
        raise AssertionError(kind)


def test_capacity_ragged_sum_form():
    # ragged form 2 L H_kv D s sum_i T_i equals the uniform form when all T_i equal T
    assert oracle.kv_bytes_ragged(32, 8, 128, 2, [4096] * 4) == oracle.kv_bytes(32, 4, 8, 128, 4096, 2)
    assert oracle.kv_bytes_ragged(1, 2, 4, 4, [3, 5]) == 2 * 1 * 2 * 4 * 4 * 8


# ---------------------------------------------------------------------------- append
@pytest.mark.parametrize("dtype", [np.uint16, np.float32])
def test_append_writes_one_slot_and_leaves_the_rest(dtype):
    B, H_kv, T_max, D = 3, 2, 9, 8
    rng = np.random.default_rng(1)
    Kc = rng.integers(0, 2**16, (B, H_kv, T_max, D)).astype(np.uint16)
    Vc = rng.integers(0, 2**16, (B, H_kv, T_max, D)).astype(np.uint16)
    if dtype == np.float32:
        Kc, Vc = _rand((B, H_kv, T_max, D), 2), _rand((B, H_kv, T_max, D), 3)
    k_new = np.ascontiguousarray(Kc[:, :, 0, :] + 1).astype(dtype) if dtype == np.uint16 else _rand((B, H_kv, D), 4)
    v_new = np.ascontiguousarray(Vc[:, :, 0, :] + 2).astype(dtype) if dtype == np.uint16 else _rand((B, H_kv, D), 5)
    lens = np.array([1, 5, T_max], dtype=np.int32)
    K0, V0 = Kc.copy(), Vc.copy()
    assert oracle.append(Kc, Vc, k_new, v_new, lens) == 0
    for b in range(B):
        s = lens[b] - 1
        assert np.array_equal(Kc[b, :, s], k_new[b]) and np.array_equal(Vc[b, :, s], v_new[b])
        keep = [t for t in range(T_max) if t != s]
        # past K/V (and untouched future slots) are bit-identical: max diff exactly 0
        assert np.array_equal(Kc[b][:, keep].view(np.uint8), K0[b][:, keep].view(np.uint8))
        assert np.array_equal(Vc[b][:, keep].view(np.uint8), V0[b][:, keep].view(np.uint8))


def test_append_rejects_out_of_range_lens():
    B, H_kv, T_max, D = 2, 1, 4, 4
    Kc = np.zeros((B, H_kv, T_max, D), np.float32)
    Vc = np.zeros_like(Kc)
    kn = np.ones((B, H_kv, D), np.float32)
    assert oracle.append(Kc, Vc, kn, kn, np.array([0, 5], np.int32)) == 2
    assert not Kc.any()


def test_prefill_write_copies_prefix():
    B, H_kv, T_in, T_max, D = 2, 2, 6, 8, 4
    K, V = _rand((B, H_kv, T_in, D), 6), _rand((B, H_kv, T_in, D), 7)
    Kc = np.zeros((B, H_kv, T_max, D), np.float32)
    Vc = np.zeros_like(Kc)
    lens = np.array([6, 3], np.int32)
    assert oracle.prefill_write(Kc, Vc, K, V, lens) == 0
    assert np.array_equal(Kc[0, :, :6], K[0]) and np.array_equal(Vc[1, :, :3], V[1, :, :3])
    assert not Kc[1, :, 3:].any() and not Kc[0, :, 6:].any()


# ---------------------------------------------------------------------------- decode attention
def test_single_slot_returns_v0_exactly():
    # softmax over one score is 1, so o = v_0
    B, H_q, H_kv, T, D = 2, 4, 2, 5, 8
    q, K, V = _rand((B, H_q, D), 1), _rand((B, H_kv, T, D), 2), _rand((B, H_kv, T, D), 3)
    out = oracle.decode_attn(q, K, V, [1, 1])
    for b in range(B):
        for j in range(H_q):
            assert np.array_equal(out[b, j], V[b, j // 2, 0].astype(np.float64))


def test_zero_query_gives_mean_of_values():
    # all scores equal => uniform weights 1/L => o = mean of the first L value rows
    B, H_q, H_kv, T, D = 2, 2, 1, 7, 16
    q = np.zeros((B, H_q, D), np.float32)
    K, V = _rand((B, H_kv, T, D), 4), _rand((B, H_kv, T, D), 5)
    lens = [7, 3]
    out = oracle.decode_attn(q, K, V, lens)
    for b in range(B):
        ref = V[b, 0, : lens[b]].astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(out[b, 0], ref, rtol=0, atol=1e-15)


def test_two_token_closed_form_pins_the_sqrt_scale():
    # q.k1 - q.k0 = sqrt(D) ln 3  =>  weights 1/4, 3/4 (a 1/D scale would give 0.366, 0.634)
    D = 4
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 1.0
    K = np.zeros((1, 1, 2, D), np.float32)
    K[0, 0, 1, 0] = math.sqrt(D) * math.log(3.0)
    V = _rand((1, 1, 2, D), 6)
    out = oracle.decode_attn(q, K, V, [2])
    s1 = float(K[0, 0, 1, 0]) / math.sqrt(D)  # the exact fp32 input, so the check is exact
    w1 = math.exp(s1) / (1 + math.exp(s1))
    ref = (1 - w1) * V[0, 0, 0].astype(np.float64) + w1 * V[0, 0, 1].astype(np.float64)
    np.testing.assert_allclose(out[0, 0], ref, rtol=0, atol=1e-14)
    np.testing.assert_allclose(out[0, 0], 0.25 * V[0, 0, 0] + 0.75 * V[0, 0, 1], atol=1e-6)


def test_gqa_map_is_floor_division():
    # value rows of KV head h are all (h+1)  =>  query head j returns floor(j/g)+1
    B, H_q, H_kv, T, D = 1, 8, 2, 6, 4
    q, K = _rand((B, H_q, D), 7), _rand((B, H_kv, T, D), 8)
    V = np.zeros((B, H_kv, T, D), np.float32)
    for h in range(H_kv):
        V[:, h] = h + 1
    out = oracle.decode_attn(q, K, V, [T])
    for j in range(H_q):
        np.testing.assert_allclose(out[0, j], j // (H_q // H_kv) + 1, rtol=1e-14)


def test_gqa_equals_mha_on_interleave_expanded_cache():
    # GQA over H_kv heads == MHA over the cache expanded with repeat_interleave (bit-identical)
    B, H_q, H_kv, T, D = 2, 6, 3, 9, 8
    q, K, V = _rand((B, H_q, D), 9), _rand((B, H_kv, T, D), 10), _rand((B, H_kv, T, D), 11)
    lens = [9, 4]
    gqa = oracle.decode_attn(q, K, V, lens)
    Ke = np.ascontiguousarray(np.repeat(K, H_q // H_kv, axis=1))
    Ve = np.ascontiguousarray(np.repeat(V, H_q // H_kv, axis=1))
    mha = oracle.decode_attn(q, Ke, Ve, lens)
    assert np.array_equal(gqa, mha)


def test_newest_slot_is_attended():
    # the last slot (the token just appended) dominates: its key is aligned with q
    D, T = 8, 6
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, :] = 1.0
    K = np.zeros((1, 1, T, D), np.float32)
    K[0, 0, T - 1, :] = 10.0
    V = _rand((1, 1, T, D), 12)
    out = oracle.decode_attn(q, K, V, [T])
    np.testing.assert_allclose(out[0, 0], V[0, 0, T - 1], atol=1e-9)


def test_slots_beyond_len_are_ignored():
    B, H_q, H_kv, T_max, D = 2, 2, 2, 10, 8
    q, K, V = _rand((B, H_q, D), 13), _rand((B, H_kv, T_max, D), 14), _rand((B, H_kv, T_max, D), 15)
    lens = [4, 7]
    a = oracle.decode_attn(q, K, V, lens)
    K2, V2 = K.copy(), V.copy()
    K2[0, :, 4:] = 1e4
    V2[0, :, 4:] = 1e4
    K2[1, :, 7:] = -1e4
    V2[1, :, 7:] = 1e4
    assert np.array_equal(a, oracle.decode_attn(q, K2, V2, lens))


def test_permutation_and_shift_invariance():
    B, H_q, H_kv, T, D = 1, 1, 1, 33, 16
    q, K, V = _rand((B, H_q, D), 16, np.float64), _rand((B, H_kv, T, D), 17, np.float64), _rand((B, H_kv, T, D), 18, np.float64)
    q32, K32, V32 = q.astype(np.float32), K.astype(np.float32), V.astype(np.float32)
    base = oracle.decode_attn(q32, K32, V32, [T])
    perm = np.random.default_rng(0).permutation(T)
    pk = np.ascontiguousarray(K32[:, :, perm])
    pv = np.ascontiguousarray(V32[:, :, perm])
    np.testing.assert_allclose(oracle.decode_attn(q32, pk, pv, [T]), base, rtol=0, atol=1e-13)
    # shifting every key by c q / |q|^2 * sqrt(D) adds c to every score: softmax unchanged
    qq = q32[0, 0].astype(np.float64)
    shift = (2.0 * math.sqrt(D) * qq / (qq @ qq)).astype(np.float32)
    Ks = np.ascontiguousarray(K32 + shift)
    np.testing.assert_allclose(oracle.decode_attn(q32, Ks, V32, [T]), base, rtol=0, atol=1e-5)


@pytest.mark.parametrize("H_q,H_kv", [(4, 4), (8, 2), (8, 1)])
def test_matches_library_sdpa_fp64(H_q, H_kv):
    # torch's scaled_dot_product_attention (CPU, fp64, one query, no mask) is a library routine
    B, T, D = 3, 21, 16
    q, K, V = _rand((B, H_q, D), 20), _rand((B, H_kv, T, D), 21), _rand((B, H_kv, T, D), 22)
    lens = [21, 13, 1]
    out = oracle.decode_attn(q, K, V, lens)
    for b in range(B):
        L = lens[b]
        qt = torch.from_numpy(q[b : b + 1].astype(np.float64)).unsqueeze(2)  # [1,H_q,1,D]
        kt = torch.from_numpy(K[b : b + 1, :, :L].astype(np.float64))
        vt = torch.from_numpy(V[b : b + 1, :, :L].astype(np.float64))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, enable_gqa=True)
        np.testing.assert_allclose(out[b], ref[0, :, 0].numpy(), rtol=0, atol=1e-12)


def test_bf16_inputs_widen_exactly():
    B, H_q, H_kv, T, D = 2, 4, 2, 12, 8
    qb = synth.queries(3, 0, B, H_q, D)
    Kb = synth.block(3, 0, "K", 0, B, H_kv, 0, T, D, B)
    Vb = synth.block(3, 0, "V", 0, B, H_kv, 0, T, D, B)
    lens = [12, 5]
    a = oracle.decode_attn(synth.bf16_bits(qb), synth.bf16_bits(Kb), synth.bf16_bits(Vb), lens)
    b = oracle.decode_attn(qb.float().numpy(), Kb.float().contiguous().numpy(), Vb.float().contiguous().numpy(), lens)
    assert np.array_equal(a, b)


def test_invalid_lens_rows_are_zero_and_counted():
    q, K, V = _rand((3, 2, 4), 30), _rand((3, 1, 5, 4), 31), _rand((3, 1, 5, 4), 32)
    out, bad = oracle.decode_attn(q, K, V, [0, 3, 6], return_bad=True)
    assert bad == 2 and not out[0].any() and not out[2].any() and out[1].any()


# ---------------------------------------------------------------------------- the layer, two ways
def _worked_example():
    cfg = {}
    for line in open(os.path.join(GOLDEN, "worked_example.txt"), encoding="utf-8"):
        if line.strip() and not line.startswith("#"):
            k, *v = line.split()
            cfg[k] = [float(x) if "e" in x or "." in x else int(x) for x in v]
    return {k: (v[0] if len(v) == 1 else v) for k, v in cfg.items()}


def test_worked_example_incremental_equals_full_recompute():
    cfg = _worked_example()
    Ws, x = synth.worked_example(cfg["seed"], cfg["hidden"], cfg["H_q"], cfg["H_kv"], cfg["D"], cfg["B"],
                                 cfg["prefill"] + cfg["decode"])
    Ws = [w.numpy() for w in Ws]
    xn = x.numpy()
    T_p, T = cfg["prefill"], cfg["prefill"] + cfg["decode"]
    inc, Kc, Vc = oracle.layer_incremental(xn, T_p, *Ws, cfg["H_q"], cfg["H_kv"], cfg["D"])
    assert list(Kc.shape) == cfg["final_cache_shape"] == list(Vc.shape)
    for step in range(cfg["decode"]):
        full, _, _ = oracle.layer_full(xn[:, : T_p + step + 1], *Ws, cfg["H_q"], cfg["H_kv"], cfg["D"])
        diff = np.abs(inc[:, step] - full[:, -1]).max()
        assert diff <= 1e-12, (step, diff)  # fp64; the pages saw ~1e-15 (rounding only)
        # the pages' own acceptance tolerance, for the record
        np.testing.assert_allclose(inc[:, step], full[:, -1], rtol=cfg["rtol"], atol=cfg["atol"])


@pytest.mark.parametrize("H_kv", [4, 2, 1])  # MHA / GQA / MQA
def test_incremental_equals_full_mha_gqa_mqa(H_kv):
    # prefill 8 then decode 12, against one full pass over 20 tokens (the W1D4 notes' check)
    hidden, H_q, D, B, T_p, T = 32, 4, 8, 2, 8, 20
    rng = np.random.default_rng(H_kv)
    WQ = rng.standard_normal((hidden, H_q * D)) / math.sqrt(hidden)
    WK = rng.standard_normal((hidden, H_kv * D)) / math.sqrt(hidden)
    WV = rng.standard_normal((hidden, H_kv * D)) / math.sqrt(hidden)
    WO = rng.standard_normal((H_q * D, hidden)) / math.sqrt(hidden)
    x = rng.standard_normal((B, T, hidden))
    inc, Kc, Vc = oracle.layer_incremental(x, T_p, WQ, WK, WV, WO, H_q, H_kv, D)
    full, Kf, Vf = oracle.layer_full(x, WQ, WK, WV, WO, H_q, H_kv, D)
    assert np.abs(inc - full[:, T_p:]).max() <= 1e-12
    # the cache the incremental path built holds exactly the full pass's K/V
    assert np.array_equal(Kc, Kf) and np.array_equal(Vc, Vf)


def test_past_kv_unchanged_by_a_longer_prefix():
    # causality: K/V of the first 12 positions are identical with 12 or 13 tokens (max diff exactly 0)
    Ws, x = synth.worked_example(T=13)
    Ws = [w.numpy() for w in Ws]
    _, K12, V12 = oracle.layer_full(x.numpy()[:, :12], *Ws, 4, 2, 4)
    _, K13, V13 = oracle.layer_full(x.numpy(), *Ws, 4, 2, 4)
    assert np.array_equal(K12, K13[:, :, :12]) and np.array_equal(V12, V13[:, :, :12])


# ---------------------------------------------------------------------------- the pins have teeth
def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_interleaved_map_is_caught():
    with oracle.planted_fault(1):
        assert _fails(test_gqa_map_is_floor_division)
        assert _fails(lambda: test_matches_library_sdpa_fp64(8, 2))


def test_planted_scale_is_caught():
    with oracle.planted_fault(2):
        assert _fails(test_two_token_closed_form_pins_the_sqrt_scale)
        assert _fails(test_worked_example_incremental_equals_full_recompute)


def test_planted_append_slot_is_caught():
    with oracle.planted_fault(3):
        assert _fails(lambda: test_append_writes_one_slot_and_leaves_the_rest(np.float32))


def test_planted_missing_new_token_is_caught():
    with oracle.planted_fault(4):
        assert _fails(test_newest_slot_is_attended)
        assert _fails(lambda: test_incremental_equals_full_mha_gqa_mqa(2))


def test_the_oracle_itself_carries_no_planted_mistakes():
    """The planted mistakes live only in the separate test build; the oracle the other tests
    trust has no switch for them."""
    import ctypes
    oracle.lib()
    assert not hasattr(ctypes.CDLL(oracle._SO), "oracle_set_fault")
    assert hasattr(ctypes.CDLL(oracle._SO_PLANTED), "oracle_set_fault")
