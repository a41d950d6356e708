"""Pins of the quantized-cache oracle (int8, one fp32 scale per (sequence, KV head, token) row;
CPU only).

The pages list int8 / fp8 caches with per-token or per-head scales as a way to read fewer bytes,
softmax accumulated in higher precision ([KVG] "KV 缓存", "MHA、GQA、MLA 与量化如何改变容量";
[M11] "11.7 KV Cache：形状、显存与带宽" §3.1 and §8).  Pinned by:

- an independent numpy restatement of the row quantizer (float32 IEEE arithmetic, round half
  to even) gives bit-identical codes and scales;
- every dequantized value is within half a quantization step of the input, and the largest
  element of a row maps to +-127;
- rows that are exactly representable (integers times a power of two, largest 127) quantize
  losslessly, and the quantized attention then equals the plain attention exactly;
- the quantized attention equals a numpy double-precision softmax over code * scale;
- appends and prefills write exactly the rows they name.
"""
import numpy as np
import pytest

import oracle


def _rand(shape, seed, dtype=np.float32):
    return np.ascontiguousarray(np.random.default_rng(seed).standard_normal(shape).astype(dtype))


def _numpy_quant(x):
    """The quantizer restated with numpy float32: scale = max|x| / 127, code = rint(x / scale)."""
    x = np.asarray(x, np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.where(scale[..., None] > 0, np.rint((x / scale[..., None]).astype(np.float32)), 0.0)
    return np.clip(c, -127, 127).astype(np.int8), scale


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_codes_and_scales_match_an_independent_restatement(dtype):
    x = _rand((50, 128), 1) * 3.0
    x[3] = 0.0                                      # an all-zero row
    x[4, :] = 1e-30                                 # tiny values
    if dtype == np.uint16:
        import torch
        xb = torch.from_numpy(x).to(torch.bfloat16)
        bits = xb.view(torch.int16).numpy().view(np.uint16)
        ref_in = xb.float().numpy()
        codes, scales = oracle.quantize_rows(np.ascontiguousarray(bits))
    else:
        ref_in = x
        codes, scales = oracle.quantize_rows(x)
    c2, s2 = _numpy_quant(ref_in)
    assert np.array_equal(scales, s2)
    assert np.array_equal(codes, c2)


def test_round_trip_within_half_a_step_and_amax_maps_to_127():
    x = _rand((200, 64), 2) * 5.0
    codes, scales = oracle.quantize_rows(x)
    deq = codes.astype(np.float64) * scales[:, None].astype(np.float64)
    assert np.all(np.abs(deq - x) <= scales[:, None] / 2 * (1 + 1e-6))
    assert np.all(np.abs(codes).max(axis=1) == 127)


def test_representable_rows_are_lossless_and_attention_is_exact():
    B, H_q, H_kv, T, D = 2, 4, 2, 9, 16
    rng = np.random.default_rng(3)
    ints = rng.integers(-127, 128, (B, H_kv, T, D)).astype(np.float32)
    ints[..., 0] = 127.0                               # the row maximum is 127 exactly
    K = ints * np.float32(2.0 ** -5)
    V = (np.roll(ints, 3, axis=-1)) * np.float32(2.0 ** -3)
    q = _rand((B, H_q, D), 4)
    lens = np.array([9, 4], np.int32)
    qc = oracle.QuantCache(B, H_kv, T, D)
    assert qc.prefill_write(np.ascontiguousarray(K), np.ascontiguousarray(V), lens) == 0
    assert np.array_equal(qc.Kq[0, :, :9].astype(np.float32) * qc.Ks[0, :, :9, None], K[0])
    got = qc.decode_attn(q, lens)
    ref = oracle.decode_attn(q, K, V, lens)
    assert np.array_equal(got, ref)


def test_attention_equals_numpy_softmax_over_dequantized_values():
    B, H_q, H_kv, T, D = 2, 6, 3, 11, 8
    K, V, q = _rand((B, H_kv, T, D), 5), _rand((B, H_kv, T, D), 6), _rand((B, H_q, D), 7)
    lens = np.array([11, 3], np.int32)
    qc = oracle.QuantCache(B, H_kv, T, D)
    assert qc.prefill_write(K, V, lens) == 0
    got = qc.decode_attn(q, lens)
    Kd = qc.Kq.astype(np.float64) * qc.Ks[..., None]
    Vd = qc.Vq.astype(np.float64) * qc.Vs[..., None]
    for b in range(B):
        for j in range(H_q):
            h = j // (H_q // H_kv)
            s = Kd[b, h, : lens[b]] @ q[b, j].astype(np.float64) / np.sqrt(D)
            p = np.exp(s - s.max())
            ref = (p / p.sum()) @ Vd[b, h, : lens[b]]
            np.testing.assert_allclose(got[b, j], ref, rtol=1e-12, atol=1e-14)


def test_append_and_prefill_write_exactly_their_rows():
    B, H_kv, T, D = 3, 2, 8, 16
    qc = oracle.QuantCache(B, H_kv, T, D)
    K, V = _rand((B, H_kv, 5, D), 8), _rand((B, H_kv, 5, D), 9)
    lens_pre = np.array([5, 0, 2], np.int32)
    assert qc.prefill_write(K, V, lens_pre) == 0
    kn, vn = _rand((B, H_kv, D), 10), _rand((B, H_kv, D), 11)
    lens = lens_pre + 1
    assert qc.append(kn, vn, lens) == 0
    c_new, s_new = oracle.quantize_rows(kn)
    c_old, s_old = oracle.quantize_rows(K)
    for b in range(B):
        assert np.array_equal(qc.Kq[b, :, lens[b] - 1], c_new[b])
        assert np.array_equal(qc.Ks[b, :, lens[b] - 1], s_new[b])
        assert np.array_equal(qc.Kq[b, :, : lens_pre[b]], c_old[b, :, : lens_pre[b]])
        assert not qc.Kq[b, :, lens[b]:].any() and not qc.Ks[b, :, lens[b]:].any()
    assert qc.append(kn, vn, np.array([0, 9, 3], np.int32)) == 2


def test_planted_scale_fault_is_caught():
    def fails(fn):
        try:
            fn()
        except AssertionError:
            return True
        return False
    with oracle.planted_fault(8):
        assert fails(lambda: test_codes_and_scales_match_an_independent_restatement(np.float32))
        assert fails(test_representable_rows_are_lossless_and_attention_is_exact)
