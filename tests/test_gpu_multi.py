"""GPU parity of decode steps with several new tokens (chunked prefill, speculative decoding):
the CUDA path through the C ABI against the oracle's lower-right causal mask.

Covers both kernels, many (group, new-token) shapes, fused and separate append, every split
count and merge path (including CTA cuts inside the new tokens, where a CTA's segment has no
visible key for some queries), launch overlap, chunked prefill of the worked example against
the dense layer, and the shapes that are refused."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import kvc, synth

from gpu_util import abs_bits, check_close, host_bits

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


class MultiCase:
    """History of lens_pre[b] tokens, T_q new tokens, q for the T_q new tokens."""

    def __init__(self, seed, B, H_q, H_kv, D, lens_pre, T_q, dtype="bf16"):
        self.B, self.H_q, self.H_kv, self.D, self.T_q = B, H_q, H_kv, D, T_q
        self.dtype = DT[dtype]
        self.lens_pre = torch.as_tensor(lens_pre, dtype=torch.int32)
        self.lens = self.lens_pre + T_q
        T_all = int(self.lens.max())
        K = synth.block(seed, 0, "K", 0, B, H_kv, 0, T_all, D, B, self.dtype)
        V = synth.block(seed, 0, "V", 0, B, H_kv, 0, T_all, D, B, self.dtype)
        self.K = K[:, :, : max(1, int(self.lens_pre.max()))].contiguous()
        self.V = V[:, :, : max(1, int(self.lens_pre.max()))].contiguous()
        self.k_new = torch.stack([K[b, :, int(lens_pre[b]) : int(lens_pre[b]) + T_q] for b in range(B)]).contiguous()
        self.v_new = torch.stack([V[b, :, int(lens_pre[b]) : int(lens_pre[b]) + T_q] for b in range(B)]).contiguous()
        self.q = synth.block(seed, 0, "Q", 0, B, H_q, 0, T_q, D, B, self.dtype).contiguous()

    def oracle(self, T_max):
        npdt = np.uint16 if self.dtype == torch.bfloat16 else np.float32
        Kc = np.zeros((self.B, self.H_kv, T_max, self.D), npdt)
        Vc = np.zeros_like(Kc)
        assert oracle.prefill_write(Kc, Vc, host_bits(self.K), host_bits(self.V), self.lens_pre.numpy()) == 0
        assert oracle.append_multi(Kc, Vc, host_bits(self.k_new), host_bits(self.v_new), self.lens.numpy()) == 0
        return oracle.decode_multi(host_bits(self.q), Kc, Vc, self.lens.numpy()), Kc, Vc

    def abs_att(self, Kc, Vc):
        """The same attention applied to |V| (bounds the weight-rounding error)."""
        return oracle.decode_multi(host_bits(self.q), Kc, np.ascontiguousarray(abs_bits(Vc)), self.lens.numpy())


def _run(case, T_max, math=0, fused=True, ctas=0, mode=-1, overlap=0):
    c = kvc.KVCache(1, case.B, case.H_q, case.H_kv, case.D, T_max,
                    "bf16" if case.dtype == torch.bfloat16 else "f32")
    try:
        c.set_math(math)
        if ctas:
            c.set_ctas(ctas)
        c.set_combine_mode(mode)
        c.set_launch_overlap(overlap)
        dev = lambda t: t.cuda()
        out = torch.full((case.B, case.H_q, case.T_q, case.D), float("nan"), dtype=case.dtype, device="cuda")
        c.prefill_write(0, dev(case.K), dev(case.V), dev(case.lens_pre))
        if fused:
            c.decode_step_multi(0, dev(case.q), dev(case.k_new), dev(case.v_new), out, dev(case.lens))
        else:
            c.append_multi(0, dev(case.k_new), dev(case.v_new), dev(case.lens))
            c.decode_attn_multi(0, dev(case.q), out, dev(case.lens))
        st, detail = c.last_error()
        assert st == kvc.KVC_OK, (st, detail)
        Kv, Vv = c.layer_views(0)
        return out, Kv.cpu(), Vv.cpu()
    finally:
        c.close()


SHAPES = [(1, 4), (4, 2), (4, 8), (8, 4), (1, 32), (2, 16)]  # (G, T_q)
PATHS = [("bf16", 128, 3), ("bf16", 128, 1), ("f32", 64, 0)]


@pytest.mark.parametrize("dtype,D,math", PATHS)
@pytest.mark.parametrize("G,T_q", SHAPES)
def test_multi_decode_matches_oracle(dtype, D, math, G, T_q):
    H_kv = 2
    case = MultiCase(900 + G * T_q + D, 3, G * H_kv, H_kv, D, [0, 37, 600], T_q, dtype)
    T_max = 700
    out, Kg, Vg = _run(case, T_max, math=math)
    ref, Kc, Vc = case.oracle(T_max)
    check_close(out, ref, case.dtype, f"multi {dtype} D={D} math={math} G={G} T_q={T_q}",
                abs_att=case.abs_att(Kc, Vc))
    assert np.array_equal(host_bits(Kg), Kc) and np.array_equal(host_bits(Vg), Vc)


@pytest.mark.parametrize("math", [3, 1])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("ctas", [1, 3, 7, 152, 600])
def test_multi_split_t_any_split_matches(ctas, mode, math):
    # one long stream and one whose history is shorter than a tile
    case = MultiCase(81, 2, 16, 2, 128, [1500, 5], 4, "bf16")
    T_max = 1600
    out, _, _ = _run(case, T_max, math=math, ctas=ctas, mode=mode)
    ref, Kc, Vc = case.oracle(T_max)
    check_close(out, ref, case.dtype, f"multi ctas={ctas} mode={mode} math={math}", abs_att=case.abs_att(Kc, Vc))


@pytest.mark.parametrize("overlap", [0, 1])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("math", [3, 1])
def test_multi_fused_separate_and_overlap(math, fused, overlap):
    case = MultiCase(82, 4, 32, 8, 128, [3000, 127, 128, 4000], 4, "bf16")
    T_max = 4100
    out, Kg, Vg = _run(case, T_max, math=math, fused=fused, overlap=overlap)
    ref, Kc, Vc = case.oracle(T_max)
    check_close(out, ref, case.dtype, f"multi fused={fused} overlap={overlap} math={math}",
                abs_att=case.abs_att(Kc, Vc))
    assert np.array_equal(host_bits(Kg), Kc) and np.array_equal(host_bits(Vg), Vc)


@pytest.mark.parametrize("chunk", [1, 2, 4, 8])
def test_chunked_prefill_of_the_worked_example_matches_the_dense_layer(chunk):
    """The glossary page's example layer (hidden 16, H_q 4, H_kv 2, D 4, fp32, seed 7), fed in
    chunks of `chunk` tokens through kvc_decode_step_multi: each chunk's projected outputs match
    the dense causal layer within the page's tolerance."""
    B, hidden, H_q, H_kv, D, T = 1, 16, 4, 2, 4, 13
    Ws, x = synth.worked_example(7, hidden, H_q, H_kv, D, B, T)
    WQ, WK, WV, WO = Ws
    full, _, _ = oracle.layer_full(x.numpy(), *[w.numpy() for w in Ws], H_q, H_kv, D)
    q_all = (x @ WQ).view(B, T, H_q, D).transpose(1, 2).contiguous()
    k_all = (x @ WK).view(B, T, H_kv, D).transpose(1, 2).contiguous()
    v_all = (x @ WV).view(B, T, H_kv, D).transpose(1, 2).contiguous()
    c = kvc.KVCache(1, B, H_q, H_kv, D, T, "f32")
    try:
        for c0 in range(0, T, chunk):
            n = min(chunk, T - c0)
            if n & (n - 1):  # the tail chunk must be a power of two too: split it
                n = 1 << (n.bit_length() - 1)
            c1 = c0 + n
            lens = torch.tensor([c1], dtype=torch.int32, device="cuda")
            out = torch.empty(B, H_q, n, D, device="cuda")
            c.decode_step_multi(0, q_all[:, :, c0:c1].contiguous().cuda(), k_all[:, :, c0:c1].contiguous().cuda(),
                                v_all[:, :, c0:c1].contiguous().cuda(), out, lens)
            y = out.cpu().permute(0, 2, 1, 3).reshape(B, n, H_q * D) @ WO
            np.testing.assert_allclose(y.numpy(), full[:, c0:c1], rtol=1e-4, atol=1e-5)
            if c1 < min(T, c0 + chunk):  # feed the rest of an uneven tail one token at a time
                for t in range(c1, min(T, c0 + chunk)):
                    lens = torch.tensor([t + 1], dtype=torch.int32, device="cuda")
                    o1 = torch.empty(B, H_q, 1, D, device="cuda")
                    c.decode_step_multi(0, q_all[:, :, t : t + 1].contiguous().cuda(),
                                        k_all[:, :, t : t + 1].contiguous().cuda(),
                                        v_all[:, :, t : t + 1].contiguous().cuda(), o1, lens)
                    y1 = o1.cpu().permute(0, 2, 1, 3).reshape(B, 1, H_q * D) @ WO
                    np.testing.assert_allclose(y1.numpy(), full[:, t : t + 1], rtol=1e-4, atol=1e-5)
        assert c.last_error() == (kvc.KVC_OK, 0)
    finally:
        c.close()


def test_multi_refuses_unsupported_shapes():
    c = kvc.KVCache(1, 2, 8, 2, 128, 64, "bf16")
    r = kvc.RollingKVCache(1, 2, 8, 2, 128, 64, "bf16")
    try:
        q = torch.zeros(2, 8, 3, 128, dtype=torch.bfloat16, device="cuda")
        out = torch.zeros_like(q)
        lens = torch.full((2,), 10, dtype=torch.int32, device="cuda")
        with pytest.raises(kvc.KvcError) as e:
            c.decode_attn_multi(0, q, out, lens)       # T_q = 3: not a power of two
        assert e.value.status == kvc.KVC_EUNSUPPORTED
        q16 = torch.zeros(2, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(kvc.KvcError) as e:
            c.decode_attn_multi(0, q16, torch.zeros_like(q16), lens)  # 4 x 16 rows > 32
        assert e.value.status == kvc.KVC_EUNSUPPORTED
        q2 = torch.zeros(2, 8, 2, 128, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(kvc.KvcError) as e:
            r.decode_attn_multi(0, q2, torch.zeros_like(q2), lens)   # rolling cache
        assert e.value.status == kvc.KVC_EUNSUPPORTED
        # lens shorter than the new tokens: flagged, zero rows
        bad = torch.tensor([1, 10], dtype=torch.int32, device="cuda")
        o2 = torch.full_like(q2, 5.0)
        c.decode_attn_multi(0, q2, o2, bad)
        st, detail = c.last_error()
        assert st == kvc.KVC_EDEVICE and detail & kvc.KVC_DEV_BAD_LENS
        assert not o2[0].float().abs().sum()
    finally:
        c.close()
        r.close()
