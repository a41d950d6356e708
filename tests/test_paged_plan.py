"""Split-T partition of a paged cache, checked on the CPU through the library's host copy of
the kernels' arithmetic (kvc_plan_cuts / kvc_plan_stream_ctas; no GPU needed).

A paged cache rounds every CTA cut down to a block boundary of the stream it falls in, so each
segment starts on a block and a 128-token tile covers whole blocks.  Checked here by brute force
over the cuts: cuts increase strictly (no empty CTA), interior cuts sit on block boundaries,
the first / last CTA of every stream match the formula the merge uses, and the partial-state
slot (CTA + stream) is injective.
"""
import ctypes

import numpy as np
import pytest

from kv_cache_decode_kvc_gb300 import kvc


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return kvc.load()


def _plan(lib, lens, H_kv, T_max, bs, P, min_tokens):
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    cuts = np.zeros(P + 1, np.int64)
    Pu = lib.kvc_plan_cuts(lens.ctypes.data, len(lens), H_kv, T_max, bs, P, min_tokens, cuts.ctypes.data)
    return Pu, cuts[: Pu + 1] if Pu > 0 else cuts[:0]


def _streams(lens, H_kv, T_max):
    """(b, h, start, L) of every non-empty stream in position order."""
    out, pos = [], 0
    for b, L in enumerate(lens):
        L = int(L) if 1 <= L <= T_max else 0
        for h in range(H_kv):
            if L:
                out.append((b, h, pos, L))
            pos += L
    return out, pos


CASES = [  # lens, H_kv, T_max, bs, P, min_tokens
    ([3001, 4500, 5999, 3000, 4200], 8, 6016, 16, 152, 256),
    ([3001, 4500, 5999, 3000, 4200], 8, 6016, 64, 152, 256),
    ([4097] * 4, 8, 4224, 128, 152, 1),
    ([131073], 1, 131328, 256, 152, 256),
    ([5, 0, 17, 300, 1], 2, 320, 16, 600, 1),     # ragged, an invalid row, tiny streams
    ([20, 700, 33], 4, 768, 32, 7, 1),
    ([1, 1, 1], 8, 16, 16, 152, 1),               # W < bs: one CTA
]


@pytest.mark.parametrize("lens,H_kv,T_max,bs,P,min_tokens", CASES)
def test_paged_cuts_are_block_aligned_and_non_empty(lib, lens, H_kv, T_max, bs, P, min_tokens):
    Pu, cuts = _plan(lib, lens, H_kv, T_max, bs, P, min_tokens)
    streams, W = _streams(lens, H_kv, T_max)
    assert 1 <= Pu <= P
    assert cuts[0] == 0 and cuts[-1] == W
    assert np.all(np.diff(cuts) > 0), "an empty CTA range"
    for c in cuts[1:-1]:
        owner = next((s, L) for (_, _, s, L) in streams if s <= c < s + L)
        assert (c - owner[0]) % bs == 0, f"cut {c} not on a block boundary"


@pytest.mark.parametrize("lens,H_kv,T_max,bs,P,min_tokens", CASES)
def test_stream_first_last_cta_match_brute_force(lib, lens, H_kv, T_max, bs, P, min_tokens):
    Pu, cuts = _plan(lib, lens, H_kv, T_max, bs, P, min_tokens)
    streams, _ = _streams(lens, H_kv, T_max)
    arr = np.ascontiguousarray(lens, dtype=np.int32)
    slots = set()
    for b, h, s, L in streams:
        holders = [i for i in range(Pu) if cuts[i] < s + L and cuts[i + 1] > s]
        f, l = ctypes.c_int(), ctypes.c_int()
        assert lib.kvc_plan_stream_ctas(arr.ctypes.data, len(arr), H_kv, T_max, bs, P, min_tokens, b, h,
                                        ctypes.byref(f), ctypes.byref(l)) == kvc.KVC_OK
        assert holders == list(range(f.value, l.value + 1)), (b, h)
        u = b * H_kv + h
        for i in holders:
            assert i + u not in slots
            slots.add(i + u)


def test_block_size_one_is_the_contiguous_partition(lib):
    lens, H_kv, P = [3001, 4500, 5999], 8, 152
    Pu, cuts = _plan(lib, lens, H_kv, 6000, 1, P, 256)
    W = 8 * sum(lens)
    assert Pu == min(P, -(-W // 256))
    assert list(cuts) == [i * W // Pu for i in range(Pu + 1)]
    for x in (0, 1, W // 3, W - 1):
        i = lib.kvc_plan_cta_of(x, W, Pu)
        assert cuts[i] <= x < cuts[i + 1]


def test_paged_create_rejects_bad_geometry_before_touching_the_device(lib):
    h = ctypes.c_void_p(123)
    # block size not in {16, 32, 64, 128, 256}
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 64, 48, 2, 4, 8, 2, 128, kvc.KVC_BF16) == kvc.KVC_EUNSUPPORTED
    assert h.value is None
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 0, 16, 2, 4, 8, 2, 128, kvc.KVC_BF16) == kvc.KVC_EINVAL
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 64, 16, 2, 0, 8, 2, 128, kvc.KVC_BF16) == kvc.KVC_EINVAL
    assert lib.kvc_create_paged(ctypes.byref(h), 1, 64, 256, 2, 1 << 23, 8, 2, 128, kvc.KVC_BF16) == kvc.KVC_ERANGE


def test_paged_calls_reject_null_handles(lib):
    assert lib.kvc_paged_decode_attn(None, 0, 1, 1, 1, 1, None) == kvc.KVC_EINVAL
    assert lib.kvc_paged_decode_step(None, 0, 1, 1, 1, 1, 1, 1, None) == kvc.KVC_EINVAL
    assert lib.kvc_paged_append(None, 0, 1, 1, 1, 1, None) == kvc.KVC_EINVAL
    assert lib.kvc_paged_prefill_write(None, 0, 1, 1, 1, 1, 1, None) == kvc.KVC_EINVAL
    assert lib.kvc_get_paged_shape(None, None, None, None) == kvc.KVC_EINVAL
