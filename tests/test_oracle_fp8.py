"""Pins of the fp8 cache oracle (E4M3 codes, one fp32 scale per (sequence, KV head, token) row;
CPU only).

The pages name fp8 beside int8 as a cache format read with the softmax accumulated in higher
precision ([M11] "11.7 KV Cache：形状、显存与带宽" §3.1 and §8; [KVG] "KV 缓存", "MHA、GQA、MLA
与量化如何改变容量").  The code is the OCP 8-bit float E4M3.  Pinned by:

- the value of each of the 256 codes equals torch's float8_e4m3fn interpretation (a library
  routine; NaN for the two NaN codes);
- every finite code encodes back to itself; every midpoint between neighbouring codes encodes
  to the even one; magnitudes beyond 448 saturate;
- on random fp32 inputs across the normal and subnormal ranges the encoder equals torch's
  round-to-nearest-even cast;
- row scales are max|x| / 448 in IEEE float32 and the codes are the torch cast of x / scale;
- the fp8 attention equals torch's fp64 scaled_dot_product_attention on value(code) * scale;
- appends and prefills write exactly the rows they name;
- each planted mistake (ties away from zero; a 240 range) makes one of these fail.
"""
import numpy as np
import pytest
import torch

import oracle

F8 = torch.float8_e4m3fn


def _torch_codes(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(F8).view(torch.uint8).numpy()


def _torch_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(F8).to(torch.float64).numpy()


def test_code_values_match_the_library():
    c = np.arange(256, dtype=np.uint8)
    v, t = oracle.e4m3_value(c), _torch_values(c)
    assert np.array_equal(np.isnan(v), np.isnan(t)) and np.isnan(v).sum() == 2
    assert np.array_equal(v[~np.isnan(v)], t[~np.isnan(t)])
    assert oracle.e4m3_value(np.uint8(0x7E)) == 448.0 and oracle.e4m3_value(np.uint8(0x01)) == 2.0 ** -9


def test_round_trip_midpoints_and_saturation():
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = oracle.e4m3_value(np.array(finite, np.uint8)).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), np.array(finite, np.uint8))
    for sign in (0, 0x80):
        for c in range(0x7E):
            a, b = oracle.e4m3_value(np.uint8(sign | c)), oracle.e4m3_value(np.uint8(sign | (c + 1)))
            mid = np.float32((a + b) / 2)  # exact: neighbouring codes differ by one quantum
            assert float(mid) == (a + b) / 2
            want = sign | (c if c % 2 == 0 else c + 1)
            assert int(oracle.e4m3_encode(mid)) == want, (hex(sign | c), float(mid))
    assert list(oracle.e4m3_encode(np.array([448.0, 449.0, 464.0, 1e30, -1e30], np.float32))) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert int(oracle.e4m3_encode(np.float32(-0.0))) == 0x80


def test_encoder_matches_the_library_cast():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(4000) * 40.0,          # normal range
                        rng.standard_normal(2000) * 2.0 ** -8,     # subnormal range
                        rng.uniform(-448.0, 448.0, 2000)]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), _torch_codes(x))


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_row_quantizer_matches_scale_and_library_cast(dtype):
    x = (np.random.default_rng(4).standard_normal((40, 128)) * 3.0).astype(np.float32)
    x[5] = 0.0
    x[6, :7] = [1e-3, -2e-3, 0, 0, 0, 0, 5e-4]
    if dtype == np.uint16:
        xb = torch.from_numpy(x).to(torch.bfloat16)
        inp = np.ascontiguousarray(xb.view(torch.int16).numpy().view(np.uint16))
        x = xb.float().numpy()
    else:
        inp = x
    codes, scales = oracle.fp8_quantize_rows(inp)
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(scales, (amax / np.float32(448.0)).astype(np.float32))
    for r in range(x.shape[0]):
        if scales[r] > 0:
            assert np.array_equal(codes[r], _torch_codes(x[r] / scales[r]))
        else:
            assert not codes[r].any()
    # the largest element of a row maps to +-448 (within one rounding of the division)
    big = np.abs(oracle.e4m3_value(codes[np.arange(40), np.abs(x).argmax(axis=1)]))
    assert np.all((big == 448.0) | (scales == 0))


def _sdpa(q, K, V, G):
    Ke = torch.from_numpy(K).repeat_interleave(G, dim=1)
    Ve = torch.from_numpy(V).repeat_interleave(G, dim=1)
    qt = torch.from_numpy(q)[:, :, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, Ke, Ve)[:, :, 0].numpy()


def test_fp8_attention_equals_the_library_on_dequantized_values():
    B, H_q, H_kv, D, T_max = 3, 8, 2, 64, 50
    rng = np.random.default_rng(5)
    K = rng.standard_normal((B, H_kv, T_max, D)).astype(np.float32)
    V = rng.standard_normal((B, H_kv, T_max, D)).astype(np.float32)
    q = rng.standard_normal((B, H_q, D)).astype(np.float32)
    lens = np.array([50, 1, 17], np.int32)
    fc = oracle.Fp8Cache(B, H_kv, T_max, D)
    assert fc.prefill_write(K, V, lens) == 0
    got = fc.decode_attn(q, lens)
    Kd = oracle.e4m3_value(fc.Kq) * fc.Ks[..., None].astype(np.float64)
    Vd = oracle.e4m3_value(fc.Vq) * fc.Vs[..., None].astype(np.float64)
    for b in range(B):
        L = lens[b]
        ref = _sdpa(q[b: b + 1].astype(np.float64), Kd[b: b + 1, :, :L], Vd[b: b + 1, :, :L], H_q // H_kv)
        assert np.max(np.abs(got[b: b + 1] - ref)) < 1e-12
    # and it is the fp8 cache's attention, not the unquantized one: they differ
    assert np.max(np.abs(got[0] - _sdpa(q[:1].astype(np.float64), K[:1].astype(np.float64),
                                        V[:1].astype(np.float64), 4)[0])) > 1e-4


def test_append_and_prefill_write_only_their_rows():
    B, H_kv, D, T_max = 2, 2, 32, 10
    rng = np.random.default_rng(6)
    K = rng.standard_normal((B, H_kv, 6, D)).astype(np.float32)
    V = rng.standard_normal((B, H_kv, 6, D)).astype(np.float32)
    fc = oracle.Fp8Cache(B, H_kv, T_max, D)
    assert fc.prefill_write(K, V, np.array([6, 3], np.int32)) == 0
    kc, ks = oracle.fp8_quantize_rows(K)
    assert np.array_equal(fc.Kq[0, :, :6], kc[0]) and np.array_equal(fc.Ks[1, :, :3], ks[1, :, :3])
    assert not fc.Kq[1, :, 3:].any() and not fc.Ks[1, :, 3:].any()
    kn = rng.standard_normal((B, H_kv, D)).astype(np.float32)
    vn = rng.standard_normal((B, H_kv, D)).astype(np.float32)
    before = fc.Kq.copy()
    assert fc.append(kn, vn, np.array([7, 4], np.int32)) == 0
    knc, _ = oracle.fp8_quantize_rows(kn)
    assert np.array_equal(fc.Kq[0, :, 6], knc[0]) and np.array_equal(fc.Kq[1, :, 3], knc[1])
    changed = np.argwhere((fc.Kq != before).any(axis=-1))
    assert {tuple(x) for x in changed} <= {(0, 0, 6), (0, 1, 6), (1, 0, 3), (1, 1, 3)}
    assert fc.append(kn, vn, np.array([0, 11], np.int32)) == 2  # invalid rows are skipped


def test_planted_ties_away_from_zero_is_caught():
    with oracle.planted_fault(9):
        with pytest.raises(AssertionError):
            test_round_trip_midpoints_and_saturation()


def test_planted_fp8_range_is_caught():
    with oracle.planted_fault(10):
        with pytest.raises(AssertionError):
            test_row_quantizer_matches_scale_and_library_cast(np.float32)
