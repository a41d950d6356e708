"""Pins of the paged-cache oracle (CPU only).

A paged cache stores each sequence's history in fixed-size blocks found through a block
table; the attention arithmetic is unchanged ([W1D4] "第 1 周 · Day 4：KV Cache 与 MQA / GQA"
§1.6; [KVG] "KV 缓存", "成本转移、失败场景与常见误解").  So every pin here ties the paged oracle
to the contiguous one (itself pinned in test_oracle_pins.py) or to plain numpy indexing:

- identity table: the pool is the contiguous cache with its token axis cut into blocks, and
  the paged result equals the contiguous result exactly (same double arithmetic, same order);
- one block per sequence: the pool is the contiguous cache itself;
- physical blocks permuted (pool and table together): identical result;
- appends and prefills land exactly where numpy fancy indexing puts them, nothing else moves;
- invalid lengths and table entries give zero rows and are counted.
"""
import numpy as np
import pytest

import oracle


def _rand(shape, seed, dtype=np.float32):
    return np.ascontiguousarray(np.random.default_rng(seed).standard_normal(shape).astype(dtype))


def _contig_to_pool(Kc, bs):
    """[B, H_kv, mb*bs, D] -> pool [B*mb, H_kv, bs, D] with the identity table."""
    B, H, T, D = Kc.shape
    mb = T // bs
    return np.ascontiguousarray(Kc.reshape(B, H, mb, bs, D).transpose(0, 2, 1, 3, 4).reshape(B * mb, H, bs, D))


def _identity_table(B, mb):
    return np.arange(B * mb, dtype=np.int32).reshape(B, mb)


def _gather(pool, table, b, h, L):
    """Rows [0, L) of (b, h) read through the table with numpy indexing."""
    bs = pool.shape[2]
    t = np.arange(L)
    return pool[table[b, t // bs], h, t % bs]


CASES = [  # B, H_q, H_kv, D, bs, mb, lens
    (3, 8, 2, 16, 4, 5, [20, 1, 13]),
    (2, 4, 4, 8, 8, 3, [24, 9]),
    (4, 6, 1, 4, 2, 7, [14, 3, 8, 1]),
]


@pytest.mark.parametrize("B,H_q,H_kv,D,bs,mb,lens", CASES)
def test_identity_table_equals_contiguous_cache(B, H_q, H_kv, D, bs, mb, lens):
    T = mb * bs
    Kc, Vc = _rand((B, H_kv, T, D), 1), _rand((B, H_kv, T, D), 2)
    q = _rand((B, H_q, D), 3)
    lens = np.array(lens, np.int32)
    ref = oracle.decode_attn(q, Kc, Vc, lens)
    got = oracle.paged_decode_attn(q, _contig_to_pool(Kc, bs), _contig_to_pool(Vc, bs),
                                   _identity_table(B, mb), lens)
    assert np.array_equal(got, ref)


def test_one_block_per_sequence_is_the_contiguous_layout():
    B, H_q, H_kv, D, T = 3, 4, 2, 8, 11
    Kc, Vc, q = _rand((B, H_kv, T, D), 4), _rand((B, H_kv, T, D), 5), _rand((B, H_q, D), 6)
    lens = np.array([11, 5, 1], np.int32)
    table = np.arange(B, dtype=np.int32).reshape(B, 1)
    assert np.array_equal(oracle.paged_decode_attn(q, Kc, Vc, table, lens),
                          oracle.decode_attn(q, Kc, Vc, lens))


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_permuted_physical_blocks_give_identical_results(dtype):
    B, H_q, H_kv, D, bs, mb = 3, 8, 2, 16, 4, 6
    nbk = B * mb + 5  # spare blocks that no sequence uses
    rng = np.random.default_rng(7)
    if dtype == np.uint16:
        pool_K = rng.integers(0x3c00, 0x4100, (nbk, H_kv, bs, D), dtype=np.uint16)
        pool_V = rng.integers(0xbc00, 0xc100, (nbk, H_kv, bs, D), dtype=np.uint16)
        q = rng.integers(0x3c00, 0x4000, (B, H_q, D), dtype=np.uint16)
    else:
        pool_K, pool_V, q = _rand((nbk, H_kv, bs, D), 8), _rand((nbk, H_kv, bs, D), 9), _rand((B, H_q, D), 10)
    table = rng.permutation(nbk)[: B * mb].astype(np.int32).reshape(B, mb)
    lens = np.array([24, 7, 13], np.int32)
    ref = oracle.paged_decode_attn(q, pool_K, pool_V, table, lens)
    perm = rng.permutation(nbk)
    K2, V2 = np.empty_like(pool_K), np.empty_like(pool_V)
    K2[perm], V2[perm] = pool_K, pool_V
    got = oracle.paged_decode_attn(q, K2, V2, perm[table].astype(np.int32), lens)
    assert np.array_equal(got, ref)
    # and the result is the contiguous attention over the gathered history
    Kc = np.zeros((B, H_kv, mb * bs, D), dtype)
    Vc = np.zeros_like(Kc)
    for b in range(B):
        for h in range(H_kv):
            Kc[b, h, : lens[b]] = _gather(pool_K, table, b, h, lens[b])
            Vc[b, h, : lens[b]] = _gather(pool_V, table, b, h, lens[b])
    assert np.array_equal(ref, oracle.decode_attn(q, Kc, Vc, lens))


def test_append_writes_exactly_one_row_per_head():
    B, H_kv, D, bs, mb = 3, 2, 8, 4, 4
    nbk = 20
    rng = np.random.default_rng(11)
    table = rng.permutation(nbk)[: B * mb].astype(np.int32).reshape(B, mb)
    Kp, Vp = _rand((nbk, H_kv, bs, D), 12), _rand((nbk, H_kv, bs, D), 13)
    K0, V0 = Kp.copy(), Vp.copy()
    kn, vn = _rand((B, H_kv, D), 14), _rand((B, H_kv, D), 15)
    lens = np.array([5, 16, 1], np.int32)
    assert oracle.paged_append(Kp, Vp, kn, vn, table, lens) == 0
    eK, eV = K0.copy(), V0.copy()
    for b in range(B):
        t = lens[b] - 1
        eK[table[b, t // bs], :, t % bs] = kn[b]
        eV[table[b, t // bs], :, t % bs] = vn[b]
    assert np.array_equal(Kp, eK) and np.array_equal(Vp, eV)


def test_prefill_then_gather_returns_the_source_rows():
    B, H_kv, D, bs, mb, T_in = 2, 3, 4, 4, 5, 19
    nbk = 12
    table = np.array([[3, 7, 0, 11, 5], [1, 9, 2, 4, 10]], np.int32)
    Kp, Vp = np.zeros((nbk, H_kv, bs, D), np.float32), np.zeros((nbk, H_kv, bs, D), np.float32)
    K, V = _rand((B, H_kv, T_in, D), 16), _rand((B, H_kv, T_in, D), 17)
    lens = np.array([19, 6], np.int32)
    assert oracle.paged_prefill_write(Kp, Vp, K, V, table, lens) == 0
    for b in range(B):
        for h in range(H_kv):
            assert np.array_equal(_gather(Kp, table, b, h, lens[b]), K[b, h, : lens[b]])
            assert np.array_equal(_gather(Vp, table, b, h, lens[b]), V[b, h, : lens[b]])
    # blocks no sequence reaches stay untouched
    used = {int(table[b, j]) for b in range(B) for j in range((lens[b] + bs - 1) // bs)}
    for e in set(range(nbk)) - used:
        assert not Kp[e].any() and not Vp[e].any()


def test_invalid_rows_are_zero_and_counted():
    B, H_q, H_kv, D, bs, mb = 4, 4, 2, 8, 4, 3
    nbk = 12
    Kp, Vp, q = _rand((nbk, H_kv, bs, D), 18), _rand((nbk, H_kv, bs, D), 19), _rand((B, H_q, D), 20)
    table = np.arange(B * mb, dtype=np.int32).reshape(B, mb)
    table[1, 1] = nbk          # out of range, needed by lens[1] = 6
    table[2, 2] = -1           # out of range but beyond lens[2] = 8: not needed, row valid
    lens = np.array([5, 6, 8, 13], np.int32)  # lens[3] > mb * bs
    out, bad = oracle.paged_decode_attn(q, Kp, Vp, table, lens, return_bad=True)
    assert bad == 2
    assert not out[1].any() and not out[3].any()
    good = [0, 2]
    Kc = np.zeros((B, H_kv, mb * bs, D), np.float32)
    Vc = np.zeros_like(Kc)
    for b in good:
        for h in range(H_kv):
            Kc[b, h, : lens[b]] = _gather(Kp, table, b, h, lens[b])
            Vc[b, h, : lens[b]] = _gather(Vp, table, b, h, lens[b])
    ref = oracle.decode_attn(q, Kc, Vc, np.where(np.isin(np.arange(B), good), lens, 0).astype(np.int32))
    assert np.array_equal(out[good], ref[good])
    kn, vn = _rand((B, H_kv, D), 21), _rand((B, H_kv, D), 22)
    K0 = Kp.copy()
    assert oracle.paged_append(Kp, Vp, kn, vn, table, lens) == 2
    assert np.array_equal(Kp[table[1, 0]], K0[table[1, 0]])  # invalid row 1 wrote nothing


def test_planted_token_major_block_is_caught():
    def fails(fn):
        try:
            fn()
        except AssertionError:
            return True
        return False
    with oracle.planted_fault(5):
        assert fails(lambda: test_identity_table_equals_contiguous_cache(*CASES[0]))
        assert fails(test_append_writes_exactly_one_row_per_head)
