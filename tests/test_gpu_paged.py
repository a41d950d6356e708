"""GPU parity of the paged cache: the CUDA path (through the C ABI) against the paged oracle.

Block tables are random permutations of a pool with spare blocks, so neighbouring logical blocks
are never neighbours in memory.  Covers every block size, the tcgen05 and CUDA-core kernels,
every split count and merge path, fused and separate append, launch overlap, bad table entries,
and a full-size 8B-GQA-shaped batch on sampled sequences."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import kvc, synth
from kv_cache_decode_kvc_gb300.workloads import WORKLOADS

from gpu_util import Case, check_close, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _table(seed, lens, bs, max_blocks, spare=5):
    """Random distinct blocks for every logical block a sequence can use; returns (table, nbk)."""
    need = len(lens) * max_blocks
    nbk = need + spare
    rng = np.random.default_rng(seed)
    table = rng.permutation(nbk)[:need].astype(np.int32).reshape(len(lens), max_blocks)
    return table, nbk


def _oracle_pool(case, table, nbk, bs):
    shape = (nbk, case.H_kv, bs, case.D)
    npdt = np.uint16 if case.dtype == torch.bfloat16 else np.float32
    Kp, Vp = np.zeros(shape, npdt), np.zeros(shape, npdt)
    assert oracle.paged_prefill_write(Kp, Vp, host_bits(case.K), host_bits(case.V), table, case.lens_pre.numpy()) == 0
    assert oracle.paged_append(Kp, Vp, host_bits(case.k_new), host_bits(case.v_new), table, case.lens.numpy()) == 0
    return Kp, Vp


def _run(case, bs, max_blocks, table, nbk, math=0, fused=True, ctas=0, mode=-1, overlap=0):
    c = kvc.PagedKVCache(1, nbk, bs, case.B, max_blocks, case.H_q, case.H_kv, case.D,
                         "bf16" if case.dtype == torch.bfloat16 else "f32")
    try:
        c.set_math(math)
        if ctas:
            c.set_ctas(ctas)
        c.set_combine_mode(mode)
        c.set_launch_overlap(overlap)
        d = case.to_device()
        tab = torch.from_numpy(table).cuda()
        out = torch.full((case.B, case.H_q, case.D), float("nan"), dtype=case.dtype, device="cuda")
        c.prefill_write(0, d["K"], d["V"], tab, d["lens_pre"])
        if fused:
            c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, tab, d["lens"])
        else:
            c.append(0, d["k_new"], d["v_new"], tab, d["lens"])
            c.decode_attn(0, d["q"], out, tab, d["lens"])
        st, detail = c.last_error()
        assert st == kvc.KVC_OK, (st, detail)
        Kv, Vv = c.layer_views(0)
        return out, Kv.cpu(), Vv.cpu()
    finally:
        c.close()


# bf16 D = 128 runs tcgen05 (3) and CUDA cores (1); other shapes CUDA cores
PATHS = [("bf16", 128, 3), ("bf16", 128, 1), ("bf16", 64, 0), ("bf16", 256, 0), ("f32", 128, 0), ("f32", 4, 0)]


@pytest.mark.parametrize("dtype,D,math", PATHS)
@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("G", [1, 4, 32])
def test_paged_decode_matches_oracle(dtype, D, math, bs, G):
    H_kv = 2
    lens_pre = [0, 37, 611, 300]
    case = Case(500 + G + bs + D, 4, G * H_kv, H_kv, D, lens_pre, dtype)
    max_blocks = -(-(max(lens_pre) + 1) // bs) + 1
    table, nbk = _table(bs + G, lens_pre, bs, max_blocks)
    out, Kg, Vg = _run(case, bs, max_blocks, table, nbk, math=math)
    Kp, Vp = _oracle_pool(case, table, nbk, bs)
    ref = oracle.paged_decode_attn(host_bits(case.q), Kp, Vp, table, case.lens.numpy())
    check_close(out, ref, case.dtype, f"paged {dtype} D={D} math={math} bs={bs} G={G}")
    assert np.array_equal(host_bits(Kg), Kp) and np.array_equal(host_bits(Vg), Vp)


@pytest.mark.parametrize("math", [3, 1])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("ctas", [1, 3, 7, 152, 600])
@pytest.mark.parametrize("bs", [16, 64, 128])
def test_paged_split_t_any_split_matches(bs, ctas, mode, math):
    case = Case(60, 2, 8, 2, 128, [1500, 0], "bf16")
    max_blocks = -(-1501 // bs)
    table, nbk = _table(61, [1500, 0], bs, max_blocks)
    out, _, _ = _run(case, bs, max_blocks, table, nbk, math=math, ctas=ctas, mode=mode)
    Kp, Vp = _oracle_pool(case, table, nbk, bs)
    ref = oracle.paged_decode_attn(host_bits(case.q), Kp, Vp, table, case.lens.numpy())
    check_close(out, ref, case.dtype, f"paged ctas={ctas} mode={mode} math={math} bs={bs}")


@pytest.mark.parametrize("overlap", [0, 1])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("math", [3, 1])
def test_paged_fused_separate_and_overlap(math, fused, overlap):
    case = Case(62, 3, 32, 8, 128, [1023, 64, 2000], "bf16")
    bs, max_blocks = 64, 33
    table, nbk = _table(63, [1023, 64, 2000], bs, max_blocks)
    out, Kg, Vg = _run(case, bs, max_blocks, table, nbk, math=math, fused=fused, overlap=overlap)
    Kp, Vp = _oracle_pool(case, table, nbk, bs)
    ref = oracle.paged_decode_attn(host_bits(case.q), Kp, Vp, table, case.lens.numpy())
    check_close(out, ref, case.dtype, f"paged fused={fused} overlap={overlap} math={math}")
    assert np.array_equal(host_bits(Kg), Kp) and np.array_equal(host_bits(Vg), Vp)


@pytest.mark.parametrize("math", [3, 1])
def test_paged_bad_table_entry_is_flagged_and_contained(math):
    """An out-of-range block id needed by sequence 1: the error word says so, nothing outside
    the pool is touched, the other sequences are exact, and the bad row's append is skipped."""
    B, H_q, H_kv, D, bs, max_blocks = 3, 8, 2, 128, 32, 8
    lens_pre = [100, 150, 200]
    case = Case(64, B, H_q, H_kv, D, lens_pre, "bf16")
    table, nbk = _table(65, lens_pre, bs, max_blocks)
    good_table = table.copy()
    table[1, 4] = nbk + 1000          # block of token 128..159 of sequence 1 (its new token 150)
    c = kvc.PagedKVCache(1, nbk, bs, B, max_blocks, H_q, H_kv, D, "bf16")
    try:
        c.set_math(math)
        d = case.to_device()
        c.prefill_write(0, d["K"], d["V"], torch.from_numpy(good_table).cuda(), d["lens_pre"])
        assert c.last_error() == (kvc.KVC_OK, 0)
        before = [t.cpu().clone() for t in c.layer_views(0)]
        out = torch.zeros(B, H_q, D, dtype=torch.bfloat16, device="cuda")
        c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, torch.from_numpy(table).cuda(), d["lens"])
        st, detail = c.last_error()
        assert st == kvc.KVC_EDEVICE and detail & kvc.KVC_DEV_BAD_BLOCK
        Kp, Vp = _oracle_pool(case, good_table, nbk, bs)
        ref = oracle.paged_decode_attn(host_bits(case.q), Kp, Vp, good_table, case.lens.numpy())
        check_close(out[[0, 2]], ref[[0, 2]], torch.bfloat16, "rows beside a bad table entry")
        Kg, _ = c.layer_views(0)
        Kg = Kg.cpu()
        # rows 0 and 2 appended; row 1's new token (block table[1, 4]) was not written anywhere
        assert np.array_equal(host_bits(Kg[good_table[0, 100 // bs], :, 100 % bs]),
                              Kp[good_table[0, 100 // bs], :, 100 % bs])
        changed = (host_bits(Kg) != host_bits(before[0])).any(axis=(1, 2, 3))
        assert set(np.flatnonzero(changed)) <= {int(good_table[0, 100 // bs]), int(good_table[2, 200 // bs])}
    finally:
        c.close()


def test_paged_full_size_gqa8b_sampled():
    """The 8B-GQA serving batch (B = 24, lengths U{3000..6000}) in 16-token blocks, one layer,
    shuffled pool; sampled sequences against the oracle on their own history."""
    w = WORKLOADS["gqa8b_b24_ragged3000_6000"]
    bs = 16
    lens = w.lens()
    max_blocks = -(-int(lens.max()) // bs)
    table, nbk = _table(66, lens.tolist(), bs, max_blocks, spare=100)
    c = kvc.PagedKVCache(1, nbk, bs, w.B, max_blocks, w.H_q, w.H_kv, w.D, "bf16")
    try:
        c.set_launch_overlap(1)
        tab = torch.from_numpy(table).cuda()
        lp = w.lens_pre()
        T_in = int(lp.max())
        K = synth.block(w.seed, 0, "K", 0, w.B, w.H_kv, 0, T_in, w.D, w.B, torch.bfloat16, "cuda")
        V = synth.block(w.seed, 0, "V", 0, w.B, w.H_kv, 0, T_in, w.D, w.B, torch.bfloat16, "cuda")
        c.prefill_write(0, K, V, tab, lp.cuda())
        del K, V
        q = synth.queries(w.seed, 0, w.B, w.H_q, w.D, torch.bfloat16, "cuda")
        kn = torch.stack([synth.block(w.seed, 0, "K", b, b + 1, w.H_kv, int(lp[b]), int(lp[b]) + 1, w.D, w.B,
                                      torch.bfloat16, "cuda")[0, :, 0] for b in range(w.B)])
        vn = torch.stack([synth.block(w.seed, 0, "V", b, b + 1, w.H_kv, int(lp[b]), int(lp[b]) + 1, w.D, w.B,
                                      torch.bfloat16, "cuda")[0, :, 0] for b in range(w.B)])
        out = torch.empty(w.B, w.H_q, w.D, dtype=torch.bfloat16, device="cuda")
        c.decode_step(0, q, kn, vn, out, tab, lens.cuda())
        assert c.last_error() == (kvc.KVC_OK, 0)
        for b in (0, 9, 23):
            L = int(lens[b])
            Kb = synth.block(w.seed, 0, "K", b, b + 1, w.H_kv, 0, L, w.D, w.B, torch.bfloat16)
            Vb = synth.block(w.seed, 0, "V", b, b + 1, w.H_kv, 0, L, w.D, w.B, torch.bfloat16)
            ref = oracle.decode_attn(host_bits(q[b : b + 1].cpu()), host_bits(Kb), host_bits(Vb),
                                     np.array([L], np.int32))
            check_close(out[b : b + 1], ref, torch.bfloat16, f"paged full size b={b}")
    finally:
        c.close()
