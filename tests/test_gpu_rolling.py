"""GPU parity of the rolling cache (sliding-window attention): the CUDA path through the C ABI
against the rolling-cache oracle, whose ring state is built one position at a time.

Covers histories shorter than, equal to and longer than the window (the new token's slot in
the middle of the ring), window 1, both kernels, fused and separate append, every split count
and merge path, launch overlap, and many consecutive steps that wrap the ring."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import kvc

from gpu_util import Case, check_close, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _oracle_ring(case, W):
    """The ring after positions [0, lens[b]) were appended in order: history rows from case.K /
    case.V, the new position from k_new / v_new."""
    npdt = np.uint16 if case.dtype == torch.bfloat16 else np.float32
    Kr = np.zeros((case.B, case.H_kv, W, case.D), npdt)
    Vr = np.zeros_like(Kr)
    K, V = host_bits(case.K), host_bits(case.V)
    kn, vn = host_bits(case.k_new), host_bits(case.v_new)
    lens_pre = case.lens_pre.numpy()
    for pos in range(int(case.lens.max())):
        lens = np.minimum(pos + 1, case.lens.numpy()).astype(np.int32)  # a finished row re-writes its last
        rows_k = np.stack([K[b, :, lens[b] - 1] if lens[b] - 1 < lens_pre[b] else kn[b] for b in range(case.B)])
        rows_v = np.stack([V[b, :, lens[b] - 1] if lens[b] - 1 < lens_pre[b] else vn[b] for b in range(case.B)])
        assert oracle.rolling_append(Kr, Vr, np.ascontiguousarray(rows_k), np.ascontiguousarray(rows_v), lens) == 0
    return Kr, Vr


def _run(case, W, math=0, fused=True, ctas=0, mode=-1, overlap=0):
    c = kvc.RollingKVCache(1, case.B, case.H_q, case.H_kv, case.D, W,
                           "bf16" if case.dtype == torch.bfloat16 else "f32")
    try:
        assert kvc.kvc_get_window(c.h) == W
        c.set_math(math)
        if ctas:
            c.set_ctas(ctas)
        c.set_combine_mode(mode)
        c.set_launch_overlap(overlap)
        d = case.to_device()
        out = torch.full((case.B, case.H_q, case.D), float("nan"), dtype=case.dtype, device="cuda")
        c.prefill_write(0, d["K"], d["V"], d["lens_pre"])
        if fused:
            c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, d["lens"])
        else:
            c.append(0, d["k_new"], d["v_new"], d["lens"])
            c.decode_attn(0, d["q"], out, d["lens"])
        st, detail = c.last_error()
        assert st == kvc.KVC_OK, (st, detail)
        Kv, Vv = c.layer_views(0)
        return out, Kv.cpu(), Vv.cpu()
    finally:
        c.close()


PATHS = [("bf16", 128, 3), ("bf16", 128, 1), ("bf16", 64, 0), ("f32", 128, 0)]


@pytest.mark.parametrize("dtype,D,math", PATHS)
@pytest.mark.parametrize("W", [1, 100, 128, 300])
@pytest.mark.parametrize("G", [1, 4, 32])
def test_rolling_decode_matches_oracle(dtype, D, math, W, G):
    # lengths below, at and above the window (wrapped, new slot mid-ring)
    lens_pre = [0, W - 1, W, 2 * W + 37, 450]
    case = Case(700 + G + W + D, 5, 2 * G, 2, D, lens_pre, dtype)
    out, Kg, Vg = _run(case, W, math=math)
    Kr, Vr = _oracle_ring(case, W)
    ref = oracle.rolling_decode_attn(host_bits(case.q), Kr, Vr, case.lens.numpy())
    check_close(out, ref, case.dtype, f"rolling {dtype} D={D} math={math} W={W} G={G}")
    assert np.array_equal(host_bits(Kg), Kr) and np.array_equal(host_bits(Vg), Vr)


@pytest.mark.parametrize("math", [3, 1])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("ctas", [1, 3, 7, 152])
def test_rolling_split_t_any_split_matches(ctas, mode, math):
    W = 1000
    case = Case(71, 2, 8, 2, 128, [2600, 10], "bf16")
    out, _, _ = _run(case, W, math=math, ctas=ctas, mode=mode)
    Kr, Vr = _oracle_ring(case, W)
    ref = oracle.rolling_decode_attn(host_bits(case.q), Kr, Vr, case.lens.numpy())
    check_close(out, ref, case.dtype, f"rolling ctas={ctas} mode={mode} math={math}")


@pytest.mark.parametrize("overlap", [0, 1])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("math", [3, 1])
def test_rolling_fused_separate_and_overlap(math, fused, overlap):
    W = 256
    case = Case(72, 3, 32, 8, 128, [1000, 255, 3], "bf16")
    out, Kg, Vg = _run(case, W, math=math, fused=fused, overlap=overlap)
    Kr, Vr = _oracle_ring(case, W)
    ref = oracle.rolling_decode_attn(host_bits(case.q), Kr, Vr, case.lens.numpy())
    check_close(out, ref, case.dtype, f"rolling fused={fused} overlap={overlap} math={math}")
    assert np.array_equal(host_bits(Kg), Kr) and np.array_equal(host_bits(Vg), Vr)


@pytest.mark.parametrize("math", [3, 1])
def test_rolling_many_steps_wrap_the_ring(math):
    """300 decode steps through a 64-slot ring (each step's token from the same seeded
    generator); checked against the oracle ring every 50 steps."""
    W, B, H_q, H_kv, D, steps = 64, 2, 8, 2, 128, 300
    start = [5, 70]
    full = Case(73, B, H_q, H_kv, D, [s + steps for s in start], "bf16")  # all positions' rows
    Kall, Vall = host_bits(full.K), host_bits(full.V)
    c = kvc.RollingKVCache(1, B, H_q, H_kv, D, W, "bf16")
    try:
        c.set_math(math)
        c.set_launch_overlap(1)
        d = full.to_device()
        lens = torch.tensor(start, dtype=torch.int32)
        c.prefill_write(0, d["K"][:, :, : max(start)].contiguous(), d["V"][:, :, : max(start)].contiguous(),
                        lens.cuda())
        npdt = np.uint16
        Kr = np.zeros((B, H_kv, W, D), npdt)
        Vr = np.zeros_like(Kr)
        for pos in range(max(start)):
            ln = np.minimum(pos + 1, np.array(start)).astype(np.int32)
            oracle.rolling_append(Kr, Vr, np.ascontiguousarray(Kall[np.arange(B), :, ln - 1]),
                                  np.ascontiguousarray(Vall[np.arange(B), :, ln - 1]), ln)
        out = torch.empty(B, H_q, D, dtype=torch.bfloat16, device="cuda")
        for step in range(steps):
            lens = lens + 1
            kn = d["K"][torch.arange(B), :, (lens - 1).long()].contiguous()
            vn = d["V"][torch.arange(B), :, (lens - 1).long()].contiguous()
            c.decode_step(0, d["q"], kn, vn, out, lens.cuda())
            ln = lens.numpy()
            oracle.rolling_append(Kr, Vr, np.ascontiguousarray(Kall[np.arange(B), :, ln - 1]),
                                  np.ascontiguousarray(Vall[np.arange(B), :, ln - 1]), ln)
            if step % 50 == 49:
                ref = oracle.rolling_decode_attn(host_bits(full.q), Kr, Vr, ln)
                check_close(out, ref, torch.bfloat16, f"rolling step {step}")
        assert c.last_error() == (kvc.KVC_OK, 0)
        Kg, _ = c.layer_views(0)
        assert np.array_equal(host_bits(Kg.cpu()), Kr)
    finally:
        c.close()


def test_rolling_rejects_zero_length_and_warp_mma():
    c = kvc.RollingKVCache(1, 2, 8, 2, 128, 64, "bf16")
    try:
        with pytest.raises(kvc.KvcError):
            c.set_math(2)
        case = Case(74, 2, 8, 2, 128, [10, 10], "bf16")
        d = case.to_device()
        out = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device="cuda")
        bad = torch.tensor([11, 0], dtype=torch.int32, device="cuda")
        c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, bad)
        st, detail = c.last_error()
        assert st == kvc.KVC_EDEVICE and detail & kvc.KVC_DEV_BAD_LENS
        assert not out[1].float().abs().sum()
    finally:
        c.close()
