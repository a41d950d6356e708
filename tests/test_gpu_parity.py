"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Sizes here span several tiles and ragged tails; test_gpu_configs.py runs the full-size
workloads on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import kvc, synth

from gpu_util import Case, check_close, host_bits

pytestmark = pytest.mark.gpu

SHAPES = [("bf16", 64), ("bf16", 128), ("bf16", 256), ("f32", 4), ("f32", 64), ("f32", 128), ("f32", 256)]
GROUPS = [1, 2, 4, 8, 16, 32]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _run(case, T_max, fused=True, ctas=0, mode=-1, layers=1, layer=0, math=0, overlap=0):
    c = kvc.KVCache(layers, case.B, case.H_q, case.H_kv, case.D, T_max,
                    "bf16" if case.dtype == torch.bfloat16 else "f32")
    try:
        if ctas:
            c.set_ctas(ctas)
        c.set_combine_mode(mode)
        c.set_math(math)
        c.set_launch_overlap(overlap)
        assert c.launch_overlap() == overlap
        if math:
            assert c.math() == math
        elif case.dtype == torch.bfloat16 and case.D == 128:
            assert c.math() == 3  # bf16 caches with D = 128 default to the tcgen05 kernel
        d = case.to_device()
        out = torch.full((case.B, case.H_q, case.D), float("nan"), dtype=case.dtype, device="cuda")
        c.prefill_write(layer, d["K"], d["V"], d["lens_pre"])
        if fused:
            c.decode_step(layer, d["q"], d["k_new"], d["v_new"], out, d["lens"])
        else:
            c.append(layer, d["k_new"], d["v_new"], d["lens"])
            c.decode_attn(layer, d["q"], out, d["lens"])
        st, detail = c.last_error()
        assert st == kvc.KVC_OK, (st, detail)
        Kv, Vv = c.layer_views(layer)
        return out, Kv.cpu(), Vv.cpu()
    finally:
        c.close()


# bf16 runs every kernel that supports the shape: tcgen05 (3, D = 128), warp MMA (2), CUDA
# cores (1); fp32 is CUDA cores only
PATHS = [(dt, D, m) for dt, D in SHAPES
         for m in (((3, 2, 1) if D == 128 else (2, 1)) if dt == "bf16" else (0,))]


@pytest.mark.parametrize("dtype,D,math", PATHS)
@pytest.mark.parametrize("G", GROUPS)
def test_decode_matches_oracle(dtype, D, math, G):
    H_kv = 2
    case = Case(100 + G + D, 3, G * H_kv, H_kv, D, [0, 37, 611], dtype)
    T_max = 640
    out, _, _ = _run(case, T_max, math=math)
    check_close(out, case.oracle_out(T_max), case.dtype, f"{dtype} D={D} G={G} math={math}")


@pytest.mark.parametrize("math", [1, 2, 3])
@pytest.mark.parametrize("fused", [True, False])
def test_append_is_bit_exact_and_leaves_other_slots(fused, math):
    case = Case(7, 4, 8, 2, 128, [5, 0, 63, 64], "bf16")
    T_max = 80
    _, Kg, Vg = _run(case, T_max, fused=fused, math=math)
    Kc, Vc = case.oracle_cache(T_max)
    assert np.array_equal(host_bits(Kg), Kc)
    assert np.array_equal(host_bits(Vg), Vc)


def test_worked_example_through_the_cache():
    """The glossary page's example: one GQA layer (hidden 16, H_q 4, H_kv 2, D 4, fp32, seed 7),
    prefill 8 tokens, decode 5; each cached step matches full causal recomputation within the
    page's tolerance, the attention matches the oracle within 1e-5, and the final cache has
    shape [1, 2, 13, 4]."""
    B, hidden, H_q, H_kv, D, T_p, T = 1, 16, 4, 2, 4, 8, 13
    Ws, x = synth.worked_example(7, hidden, H_q, H_kv, D, B, T)
    WQ, WK, WV, WO = Ws
    # projections are the harness's job (fp32, CPU): q, k, v for every position
    q_all = (x @ WQ).view(B, T, H_q, D).transpose(1, 2).contiguous()   # [B,H_q,T,D]
    k_all = (x @ WK).view(B, T, H_kv, D).transpose(1, 2).contiguous()  # [B,H_kv,T,D]
    v_all = (x @ WV).view(B, T, H_kv, D).transpose(1, 2).contiguous()
    full_outs = []
    for step in range(T - T_p):
        full, _, _ = oracle.layer_full(x[:, : T_p + step + 1].numpy(), *[w.numpy() for w in Ws], H_q, H_kv, D)
        full_outs.append(full[:, -1])
    c = kvc.KVCache(1, B, H_q, H_kv, D, T, "f32")
    try:
        lens_pre = torch.tensor([T_p], dtype=torch.int32)
        c.prefill_write(0, k_all[:, :, :T_p].cuda(), v_all[:, :, :T_p].cuda(), lens_pre.cuda())
        Kc = np.zeros((B, H_kv, T, D), np.float32)
        Vc = np.zeros_like(Kc)
        oracle.prefill_write(Kc, Vc, k_all[:, :, :T_p].contiguous().numpy(), v_all[:, :, :T_p].contiguous().numpy(), lens_pre.numpy())
        for step in range(T - T_p):
            pos = T_p + step
            lens = torch.tensor([pos + 1], dtype=torch.int32)
            qt = q_all[:, :, pos].contiguous()
            kt = k_all[:, :, pos].contiguous()
            vt = v_all[:, :, pos].contiguous()
            out = torch.empty(B, H_q, D, device="cuda")
            c.decode_step(0, qt.cuda(), kt.cuda(), vt.cuda(), out, lens.cuda())
            oracle.append(Kc, Vc, kt.numpy(), vt.numpy(), lens.numpy())
            ref = oracle.decode_attn(qt.numpy(), Kc, Vc, lens.numpy())
            check_close(out, ref, torch.float32, f"worked example step {step}")
            y = out.cpu().reshape(B, 1, H_q * D) @ WO  # the harness's output projection
            np.testing.assert_allclose(y[:, 0].numpy(), full_outs[step], rtol=1e-4, atol=1e-5)
        Kv, Vv = c.layer_views(0)
        assert tuple(Kv.shape) == tuple(Vv.shape) == (1, 2, 13, 4)
        assert np.array_equal(Kv.cpu().numpy(), Kc)
        assert c.last_error() == (kvc.KVC_OK, 0)
    finally:
        c.close()


@pytest.mark.parametrize("math", [1, 2, 3])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 152, 600])
def test_split_t_any_split_matches(ctas, mode, math):
    # one long and one 1-token stream per KV head; every split count and both merge paths
    case = Case(55, 2, 8, 2, 128, [1500, 0], "bf16")
    T_max = 1600
    out, _, _ = _run(case, T_max, ctas=ctas, mode=mode, math=math)
    check_close(out, case.oracle_out(T_max), case.dtype, f"ctas={ctas} mode={mode} math={math}")


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("ctas", [3, 7, 152])
@pytest.mark.parametrize("G", [16, 32])
def test_split_t_large_groups_tcgen05(G, ctas, mode):
    # groups of 16 and 32 heads (eight softmax warps, weights stored MN-major) cut across CTAs
    case = Case(58 + G, 3, 2 * G, 2, 128, [1500, 3, 700], "bf16")
    T_max = 1600
    out, _, _ = _run(case, T_max, ctas=ctas, mode=mode, math=3)
    check_close(out, case.oracle_out(T_max), case.dtype, f"G={G} ctas={ctas} mode={mode}")


@pytest.mark.parametrize("ctas", [1, 5, 64])
def test_split_t_fp32_is_tight(ctas):
    case = Case(56, 3, 32, 1, 128, [2000, 17, 900], "f32")
    T_max = 2048
    out, _, _ = _run(case, T_max, ctas=ctas, mode=0)
    check_close(out, case.oracle_out(T_max), case.dtype, f"fp32 MQA ctas={ctas}")


@pytest.mark.parametrize("math", [1, 2, 3])
def test_maximum_length_and_single_token(math):
    case = Case(57, 2, 4, 1, 128, [255, 0], "bf16")  # lens = [T_max, 1]
    out, _, _ = _run(case, 256, math=math)
    check_close(out, case.oracle_out(256), case.dtype, "T_max edge")
    # a 1-token history returns v_new exactly (softmax of one score is 1)
    assert torch.equal(out[1].cpu(), case.v_new[1, 0].expand(4, 128))


@pytest.mark.parametrize("math", [1, 2, 3])
def test_invalid_lengths_flag_and_zero_rows(math):
    B, H_q, H_kv, D, T_max = 4, 8, 2, 128, 64
    case = Case(58, B, H_q, H_kv, D, [10, 20, 30, 40], "bf16")
    c = kvc.KVCache(1, B, H_q, H_kv, D, T_max, "bf16")
    try:
        c.set_math(math)
        d = case.to_device()
        c.prefill_write(0, d["K"], d["V"], d["lens_pre"])
        bad = torch.tensor([11, 0, 31, T_max + 5], dtype=torch.int32, device="cuda")
        out = torch.full((B, H_q, D), 7.0, dtype=torch.bfloat16, device="cuda")
        c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, bad)
        st, detail = c.last_error()
        assert st == kvc.KVC_EDEVICE and detail & kvc.KVC_DEV_BAD_LENS
        assert c.last_error() == (kvc.KVC_OK, 0)  # cleared
        assert not out[1].float().abs().sum() and not out[3].float().abs().sum()
        ref = case.oracle_out(T_max)
        check_close(out[[0, 2]], ref[[0, 2]], torch.bfloat16, "valid rows beside invalid ones")
        # the invalid rows appended nothing
        Kv, _ = c.layer_views(0)
        Kc, _ = case.oracle_cache(T_max)
        assert np.array_equal(host_bits(Kv[[0, 2]].cpu()), Kc[[0, 2]])
        assert not Kv[1, :, 20].float().abs().sum()  # slot lens_pre[1] untouched (was never written)
    finally:
        c.close()


@pytest.mark.parametrize("math", [1, 2, 3])
def test_repeated_steps_reuse_workspace(math):
    # the arrival counters must be back at zero after every call
    case = Case(59, 2, 16, 2, 128, [3000, 2999], "bf16")
    T_max = 3001
    c = kvc.KVCache(1, 2, 16, 2, 128, T_max, "bf16")
    try:
        c.set_combine_mode(0)
        c.set_math(math)
        d = case.to_device()
        c.prefill_write(0, d["K"], d["V"], d["lens_pre"])
        ref = case.oracle_out(T_max)
        for _ in range(5):
            out = torch.empty(2, 16, 128, dtype=torch.bfloat16, device="cuda")
            c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, d["lens"])
            check_close(out, ref, torch.bfloat16, "repeat")
        assert c.last_error() == (kvc.KVC_OK, 0)
    finally:
        c.close()


def test_generator_is_device_independent():
    a = synth.block(3, 5, "V", 2, 6, 4, 100, 357, 128, 8, torch.bfloat16, "cpu")
    b = synth.block(3, 5, "V", 2, 6, 4, 100, 357, 128, 8, torch.bfloat16, "cuda")
    assert torch.equal(a, b.cpu())


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("ctas", [3, 152])
@pytest.mark.parametrize("G", [1, 4, 32])
def test_launch_overlap_gives_the_same_results(G, ctas, fused):
    """Early history loads (before the preceding grid completes) change no result: every
    (stream, tile) layout, including tiles holding a stream's new row, which are loaded only
    after the wait."""
    case = Case(300 + G, 3, 2 * G, 2, 128, [700, 0, 129], "bf16")
    T_max = 800
    out, Kg, Vg = _run(case, T_max, fused=fused, ctas=ctas, math=3, overlap=1)
    check_close(out, case.oracle_out(T_max), case.dtype, f"overlap G={G} ctas={ctas}")
    Kc, Vc = case.oracle_cache(T_max)
    assert np.array_equal(host_bits(Kg), Kc) and np.array_equal(host_bits(Vg), Vc)


def test_launch_overlap_layer_loop_matches_oracle():
    """A decode step over several layers back to back on one stream with overlap on: each
    launch starts loading while the previous layer's launch is finishing."""
    B, H_q, H_kv, D, T_max, L = 4, 32, 8, 128, 1200, 6
    lens_pre = [1100, 5, 640, 999]
    cases = [Case(400 + l, B, H_q, H_kv, D, lens_pre, "bf16", layer=l) for l in range(L)]
    c = kvc.KVCache(L, B, H_q, H_kv, D, T_max, "bf16")
    try:
        c.set_math(3)
        c.set_launch_overlap(1)
        devs = [cs.to_device() for cs in cases]
        for l, d in enumerate(devs):
            c.prefill_write(l, d["K"], d["V"], d["lens_pre"])
        outs = [torch.full((B, H_q, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        for _ in range(3):  # repeated steps: the same token re-appended, same outputs
            for l, d in enumerate(devs):
                c.decode_step(l, d["q"], d["k_new"], d["v_new"], outs[l], d["lens"])
        assert c.last_error() == (kvc.KVC_OK, 0)
        for l in range(L):
            check_close(outs[l], cases[l].oracle_out(T_max), torch.bfloat16, f"layer {l}")
    finally:
        c.close()
