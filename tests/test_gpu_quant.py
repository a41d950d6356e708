"""GPU parity of the int8 cache (one fp32 scale per (sequence, KV head, token) row): the CUDA
path through the C ABI against the quantized-cache oracle.

The codes and scales the GPU writes (prefill, append, fused step) must equal the oracle's bit
for bit (both sides quantize in IEEE fp32 with round-half-even); the attention over them must
match the oracle's double-precision result within the decode tolerance and the one-ulp bar
(widened by the weight-rounding bound, see gpu_util.check_close)."""
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


def _oracle(case, T_max):
    qc = oracle.QuantCache(case.B, case.H_kv, T_max, case.D)
    assert qc.prefill_write(host_bits(case.K), host_bits(case.V), case.lens_pre.numpy()) == 0
    assert qc.append(host_bits(case.k_new), host_bits(case.v_new), case.lens.numpy()) == 0
    return qc


def _abs_att(case, qc):
    """The same attention on |code| * scale: bounds the weight-rounding error."""
    a = oracle.QuantCache(case.B, case.H_kv, qc.Kq.shape[2], case.D)
    a.Kq[...] = qc.Kq
    a.Ks[...] = qc.Ks
    a.Vq[...] = np.abs(qc.Vq.astype(np.int16)).astype(np.int8)
    a.Vs[...] = qc.Vs
    return a.decode_attn(host_bits(case.q), case.lens.numpy())


def _run(case, T_max, fused=True, ctas=0, mode=-1, overlap=0):
    c = kvc.QuantKVCache(1, case.B, case.H_q, case.H_kv, case.D, T_max)
    try:
        if ctas:
            c.set_ctas(ctas)
        c.set_combine_mode(mode)
        c.set_launch_overlap(overlap)
        assert c.math() == 3
        d = case.to_device()
        out = torch.full((case.B, case.H_q, case.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        c.prefill_write(0, d["K"], d["V"], d["lens_pre"])
        if fused:
            c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, d["lens"])
        else:
            c.append(0, d["k_new"], d["v_new"], d["lens"])
            c.decode_attn(0, d["q"], out, d["lens"])
        st, detail = c.last_error()
        assert st == kvc.KVC_OK, (st, detail)
        return out, [t.cpu() for t in c.layer_views(0)]
    finally:
        c.close()


def _check_cache(views, qc):
    Kq, Vq, Ks, Vs = views
    assert np.array_equal(Kq.numpy(), qc.Kq) and np.array_equal(Vq.numpy(), qc.Vq)
    assert np.array_equal(Ks.numpy().view(np.uint32), qc.Ks.view(np.uint32))
    assert np.array_equal(Vs.numpy().view(np.uint32), qc.Vs.view(np.uint32))


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("fused", [True, False])
def test_quant_decode_matches_oracle(G, fused):
    H_kv = 2
    case = Case(1000 + G, 4, G * H_kv, H_kv, 128, [0, 37, 611, 300], "bf16")
    T_max = 640
    out, views = _run(case, T_max, fused=fused)
    qc = _oracle(case, T_max)
    _check_cache(views, qc)
    ref = qc.decode_attn(host_bits(case.q), case.lens.numpy())
    check_close(out, ref, torch.bfloat16, f"int8 G={G} fused={fused}", abs_att=_abs_att(case, qc))


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("ctas", [1, 3, 7, 152, 600])
def test_quant_split_t_any_split_matches(ctas, mode):
    case = Case(1010, 2, 8, 2, 128, [1500, 0], "bf16")
    T_max = 1600
    out, _ = _run(case, T_max, ctas=ctas, mode=mode)
    qc = _oracle(case, T_max)
    ref = qc.decode_attn(host_bits(case.q), case.lens.numpy())
    check_close(out, ref, torch.bfloat16, f"int8 ctas={ctas} mode={mode}", abs_att=_abs_att(case, qc))


@pytest.mark.parametrize("G", [1, 8])
@pytest.mark.parametrize("ctas", [1, 2])
def test_quant_long_segments_per_cta(G, ctas):
    """One or two CTAs, so each streams dozens of tiles through every ring stage and both
    tensor-memory K buffers many times over (G = 8 runs the four-converter layout, G = 1 the
    eight-converter one with its own MMA2 warp); one stream ends in a partial tile."""
    case = Case(1020 + G, 3, 2 * G, 2, 128, [2000, 1333, 129], "bf16")
    T_max = 2048
    out, views = _run(case, T_max, ctas=ctas)
    qc = _oracle(case, T_max)
    _check_cache(views, qc)
    ref = qc.decode_attn(host_bits(case.q), case.lens.numpy())
    check_close(out, ref, torch.bfloat16, f"int8 long G={G} ctas={ctas}", abs_att=_abs_att(case, qc))


@pytest.mark.parametrize("overlap", [0, 1])
def test_quant_layer_loop_with_overlap(overlap):
    """Several layers back to back (each with its own seeded data), repeated steps."""
    B, H_q, H_kv, D, T_max, L = 3, 32, 8, 128, 2100, 4
    lens_pre = [2000, 5, 1024]
    cases = [Case(1020 + l, B, H_q, H_kv, D, lens_pre, "bf16", layer=l) for l in range(L)]
    c = kvc.QuantKVCache(L, B, H_q, H_kv, D, T_max)
    try:
        c.set_launch_overlap(overlap)
        devs = [cs.to_device() for cs in cases]
        for l, d in enumerate(devs):
            c.prefill_write(l, d["K"], d["V"], d["lens_pre"])
        outs = [torch.empty(B, H_q, D, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        for _ in range(2):
            for l, d in enumerate(devs):
                c.decode_step(l, d["q"], d["k_new"], d["v_new"], outs[l], d["lens"])
        assert c.last_error() == (kvc.KVC_OK, 0)
        for l in range(L):
            qc = _oracle(cases[l], T_max)
            _check_cache([t.cpu() for t in c.layer_views(l)], qc)
            ref = qc.decode_attn(host_bits(cases[l].q), cases[l].lens.numpy())
            check_close(outs[l], ref, torch.bfloat16, f"int8 layer {l}", abs_att=_abs_att(cases[l], qc))
    finally:
        c.close()


def test_quant_full_size_gqa8b_sampled():
    """The 8B-GQA serving batch (B = 24, lengths U{3000..6000}) in an int8 cache, one layer;
    sampled sequences against the oracle on their own quantized history."""
    w = WORKLOADS["gqa8b_b24_ragged3000_6000"]
    lp, lens = w.lens_pre(), w.lens()
    c = kvc.QuantKVCache(1, w.B, w.H_q, w.H_kv, w.D, w.T_max())
    try:
        c.set_launch_overlap(1)
        T_in = int(lp.max())
        K = synth.block(w.seed, 0, "K", 0, w.B, w.H_kv, 0, T_in, w.D, w.B, torch.bfloat16, "cuda")
        V = synth.block(w.seed, 0, "V", 0, w.B, w.H_kv, 0, T_in, w.D, w.B, torch.bfloat16, "cuda")
        c.prefill_write(0, K, V, lp.cuda())
        del K, V
        q = synth.queries(w.seed, 0, w.B, w.H_q, w.D, torch.bfloat16, "cuda")
        kn = torch.stack([synth.block(w.seed, 0, "K", b, b + 1, w.H_kv, int(lp[b]), int(lp[b]) + 1, w.D, w.B,
                                      torch.bfloat16, "cuda")[0, :, 0] for b in range(w.B)])
        vn = torch.stack([synth.block(w.seed, 0, "V", b, b + 1, w.H_kv, int(lp[b]), int(lp[b]) + 1, w.D, w.B,
                                      torch.bfloat16, "cuda")[0, :, 0] for b in range(w.B)])
        out = torch.empty(w.B, w.H_q, w.D, dtype=torch.bfloat16, device="cuda")
        c.decode_step(0, q, kn, vn, out, lens.cuda())
        assert c.last_error() == (kvc.KVC_OK, 0)
        for b in (0, 11, 23):
            L = int(lens[b])
            Kb = synth.block(w.seed, 0, "K", b, b + 1, w.H_kv, 0, L, w.D, w.B, torch.bfloat16)
            Vb = synth.block(w.seed, 0, "V", b, b + 1, w.H_kv, 0, L, w.D, w.B, torch.bfloat16)
            qc = oracle.QuantCache(1, w.H_kv, L, w.D)
            assert qc.prefill_write(host_bits(Kb), host_bits(Vb), np.array([L], np.int32)) == 0
            ref = qc.decode_attn(host_bits(q[b : b + 1].cpu()), np.array([L], np.int32))
            check_close(out[b : b + 1], ref, torch.bfloat16, f"int8 full size b={b}", tight=False)
    finally:
        c.close()


def test_quant_refuses_what_it_cannot_run():
    with pytest.raises(kvc.KvcError) as e:
        kvc.QuantKVCache(1, 2, 32, 2, 128, 64)      # 16 query heads per KV head
    assert e.value.status == kvc.KVC_EUNSUPPORTED
    with pytest.raises(kvc.KvcError) as e:
        kvc.QuantKVCache(1, 2, 8, 2, 64, 64)        # D = 64
    assert e.value.status == kvc.KVC_EUNSUPPORTED
    c = kvc.QuantKVCache(1, 2, 8, 2, 128, 64)
    try:
        with pytest.raises(kvc.KvcError):
            c.set_math(1)
        bad = torch.tensor([0, 65], dtype=torch.int32, device="cuda")
        case = Case(1030, 2, 8, 2, 128, [10, 10], "bf16")
        d = case.to_device()
        out = torch.full((2, 8, 128), 3.0, dtype=torch.bfloat16, device="cuda")
        c.decode_step(0, d["q"], d["k_new"], d["v_new"], out, bad)
        st, detail = c.last_error()
        assert st == kvc.KVC_EDEVICE and detail & kvc.KVC_DEV_BAD_LENS
        assert not out.float().abs().sum()
    finally:
        c.close()
