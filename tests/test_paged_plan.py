"""Split-T partition of the attention kernels, checked on the CPU through the library's host
copy of the kernels' arithmetic (kvc_plan_cuts / kvc_plan_stream_ctas; no GPU needed), and the
paged cache's host-side argument checks.

Each stream is cut into units of g tokens (g = 128, one tcgen05 tile; g = 1, the plain token
split, or a paged block, for groups of 16 or 32 heads merged inside the kernel; the last unit of
a stream may be partial); with g = 128 a stream is charged one more unit for its start, placed
before its first token unit.  CTA i of Pu takes units [floor(i U / Pu), floor((i+1) U / Pu)).
Checked here: the cuts equal those of a separate Python statement of that rule, never decrease
and sit on unit boundaries of their stream (so on block boundaries of a paged pool with blocks
of up to 128 tokens); the first / last CTA of every stream match a brute-force search over the
cuts; the partial-state slot (CTA + stream) is injective.
"""
import ctypes

import numpy as np
import pytest

from kv_cache_decode_kvc_gb300 import kvc

UNIT = 128


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return kvc.load()


def _plan(lib, lens, H_kv, T_max, P, min_tokens, grain=UNIT):
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    cuts = np.zeros(P + 1, np.int64)
    Pu = lib.kvc_plan_cuts(lens.ctypes.data, len(lens), H_kv, T_max, grain, P, min_tokens, cuts.ctypes.data)
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


def _units_in(streams, a, b, g=UNIT):
    """Units (g-token pieces of a stream, the last one partial) that meet positions [a, b)."""
    n = 0
    for _, _, s, L in streams:
        lo, hi = max(a, s), min(b, s + L)
        if lo < hi:
            n += (hi - s + g - 1) // g - (lo - s) // g
    return n


def _model_cuts(lens, H_kv, T_max, P, min_tokens, g):
    """The partition rule, restated: stream costs, unit cuts, token positions."""
    streams, W = _streams(lens, H_kv, T_max)
    c = 1 if g == UNIT else 0
    costs = [(L + g - 1) // g + c for *_, L in streams]
    cs = np.concatenate([[0], np.cumsum(costs)])
    U = int(cs[-1])
    Pu = min(P, -(-W // min_tokens), U)

    def pos(x):
        k = int(np.searchsorted(cs, x, side="right") - 1)
        j = x - cs[k]
        return streams[k][2] + max(0, j - c) * g

    return Pu, [pos(i * U // Pu) for i in range(Pu)] + [W]


CASES = [  # lens, H_kv, T_max, P, min_tokens
    ([3001, 4500, 5999, 3000, 4200], 8, 6016, 152, 256),
    ([4097] * 4, 8, 4224, 152, 1),               # every stream ends in a one-token unit
    ([4097], 32, 4097, 152, 256),                # one sequence of 32 streams
    ([131073], 1, 131328, 152, 256),             # one long stream
    ([5, 0, 17, 300, 1], 2, 320, 600, 1),        # ragged, an invalid row, tiny streams
    ([20, 700, 33], 4, 768, 7, 1),
    ([1, 1, 1], 8, 16, 152, 1),                  # fewer units than CTAs
    ([4000, 129, 128, 127, 257], 3, 4096, 13, 64),
]


@pytest.mark.parametrize("grain", [UNIT, 1, 32])
@pytest.mark.parametrize("lens,H_kv,T_max,P,min_tokens", CASES)
def test_cuts_fall_on_unit_boundaries_and_balance_the_units(lib, lens, H_kv, T_max, P, min_tokens, grain):
    Pu, cuts = _plan(lib, lens, H_kv, T_max, P, min_tokens, grain)
    streams, W = _streams(lens, H_kv, T_max)
    mPu, mcuts = _model_cuts(lens, H_kv, T_max, P, min_tokens, grain)
    assert Pu == mPu and list(cuts) == mcuts
    assert cuts[0] == 0 and cuts[-1] == W
    assert np.all(np.diff(cuts) >= 0)
    for c in cuts[1:-1]:
        if c == W:
            continue
        owner = next(s for (_, _, s, L) in streams if s <= c < s + L)
        assert (c - owner) % grain == 0, f"cut {c} inside a unit"
    # token units per CTA: the unit counts differ by at most one plus the stream starts held
    per_cta = [_units_in(streams, cuts[i], cuts[i + 1], grain) for i in range(Pu)]
    U_tok = sum((L + grain - 1) // grain for *_, L in streams)
    assert sum(per_cta) == U_tok


@pytest.mark.parametrize("grain", [UNIT, 1])
@pytest.mark.parametrize("lens,H_kv,T_max,P,min_tokens", CASES)
def test_stream_first_last_cta_match_brute_force(lib, lens, H_kv, T_max, P, min_tokens, grain):
    Pu, cuts = _plan(lib, lens, H_kv, T_max, P, min_tokens, grain)
    streams, _ = _streams(lens, H_kv, T_max)
    arr = np.ascontiguousarray(lens, dtype=np.int32)
    slots = set()
    for b, h, s, L in streams:
        holders = [i for i in range(Pu) if cuts[i] < s + L and cuts[i + 1] > s]
        f, l = ctypes.c_int(), ctypes.c_int()
        assert lib.kvc_plan_stream_ctas(arr.ctypes.data, len(arr), H_kv, T_max, grain, P, min_tokens, b, h,
                                        ctypes.byref(f), ctypes.byref(l)) == kvc.KVC_OK
        assert holders == list(range(f.value, l.value + 1)), (b, h)
        u = b * H_kv + h
        for i in holders:
            assert i + u not in slots
            slots.add(i + u)


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_paged_blocks_are_never_split(lib, bs):
    lens, H_kv, P = [3001, 4500, 5999, 3000, 4200], 8, 152
    T_max = -(-6000 // bs) * bs
    _, cuts = _plan(lib, lens, H_kv, T_max, P, 256)
    streams, _ = _streams(lens, H_kv, T_max)
    for c in cuts[1:-1]:
        owner = next(s for (_, _, s, L) in streams if s <= c < s + L)
        assert (c - owner) % bs == 0


def test_stream_starts_are_charged_a_unit(lib):
    # 4 streams of 4 units each, 2 CTAs: costs 5 + 5 + 5 + 5, so each CTA takes two streams
    lens, H_kv = [512, 512], 2
    Pu, cuts = _plan(lib, lens, H_kv, 512, 2, 1)
    assert Pu == 2 and list(cuts) == [0, 1024, 2048]
    # 3 CTAs over costs 5 + 5 + 5 + 5 = 20: cuts at cost 6 (stream 1, first token unit) and 13
    # (stream 2, its third unit: token 2 * 128)
    Pu, cuts = _plan(lib, lens, H_kv, 512, 3, 1)
    assert Pu == 3 and list(cuts) == [0, 512, 1024 + 256, 2048]


def test_block_size_one_grain_is_the_plain_token_split(lib):
    lens, H_kv, P = [3001, 4500, 5999], 8, 152
    Pu, cuts = _plan(lib, lens, H_kv, 6000, P, 256, grain=1)
    W = 8 * sum(lens)
    assert Pu == min(P, -(-W // 256))
    assert list(cuts) == [i * W // Pu for i in range(Pu + 1)]


def test_grain_follows_the_query_group_and_merge_mode(lib):
    assert [lib.kvc_plan_grain(G, 0, 1) for G in (1, 2, 4, 8, 16, 32)] == [UNIT] * 4 + [1, 1]
    assert [lib.kvc_plan_grain(G, 1, 1) for G in (1, 8, 16, 32)] == [UNIT] * 4
    assert [lib.kvc_plan_grain(32, 0, bs) for bs in (16, 64, 256)] == [16, 64, 256]
    assert lib.kvc_plan_grain(8, 0, 256) == UNIT
    assert lib.kvc_plan_grain(0, 0, 1) == -1 and lib.kvc_plan_grain(4, 2, 1) == -1


def test_plan_rejects_prefix_overflow_and_bad_arguments(lib):
    arr = np.ascontiguousarray([5, 5], dtype=np.int32)
    cuts = np.zeros(8, np.int64)
    assert lib.kvc_plan_cuts(arr.ctypes.data, 2, 1, 1 << 30, UNIT, 4, 1, cuts.ctypes.data) == -1  # B * T_max = 2^31
    assert lib.kvc_plan_cuts(arr.ctypes.data, 2, 1, 16, UNIT, 0, 1, cuts.ctypes.data) == -1
    assert lib.kvc_plan_cuts(arr.ctypes.data, 2, 1, 16, UNIT, 4, 0, cuts.ctypes.data) == -1
    assert lib.kvc_plan_cuts(arr.ctypes.data, 2, 1, 16, 0, 4, 1, cuts.ctypes.data) == -1
    f, l = ctypes.c_int(), ctypes.c_int()
    assert lib.kvc_plan_stream_ctas(arr.ctypes.data, 2, 1, 1 << 30, UNIT, 4, 1, 0, 0, ctypes.byref(f),
                                    ctypes.byref(l)) == kvc.KVC_ERANGE
    empty = np.ascontiguousarray([5, 0], dtype=np.int32)
    assert lib.kvc_plan_stream_ctas(empty.ctypes.data, 2, 1, 16, UNIT, 4, 1, 1, 0, ctypes.byref(f),
                                    ctypes.byref(l)) == kvc.KVC_EINVAL


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
