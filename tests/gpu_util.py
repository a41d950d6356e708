"""Helpers shared by the GPU tests: seeded inputs for both sides, oracle references,
and the tolerance checks.  Inputs come from kv_cache_decode_kvc_gb300.synth (counter-based,
identical on CPU and GPU); expected values come from the oracle only."""
import numpy as np
import torch

import oracle
from kv_cache_decode_kvc_gb300 import kvc, synth

DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Oracle input format: uint16 bf16 bits or float32."""
    t = t.contiguous().cpu()
    return synth.bf16_bits(t) if t.dtype == torch.bfloat16 else t.numpy()


def new_rows(seed, layer, tensor, lens_pre, H, D, B, dtype):
    """Row t = lens_pre[b] of every (b, head) stream: the token a step appends, [B, H, D]."""
    rows = [synth.block(seed, layer, tensor, b, b + 1, H, int(lens_pre[b]), int(lens_pre[b]) + 1, D, B,
                        dtype)[0, :, 0] for b in range(B)]
    return torch.stack(rows).contiguous()


class Case:
    """One layer's worth of seeded inputs: history of lens_pre[b] tokens, the new token, q."""

    def __init__(self, seed, B, H_q, H_kv, D, lens_pre, dtype="bf16", layer=0):
        self.seed, self.B, self.H_q, self.H_kv, self.D, self.layer = seed, B, H_q, H_kv, D, layer
        self.dtype = DT[dtype]
        self.lens_pre = torch.as_tensor(lens_pre, dtype=torch.int32)
        self.lens = self.lens_pre + 1
        self.T_in = max(1, int(self.lens_pre.max()))
        self.K = synth.block(seed, layer, "K", 0, B, H_kv, 0, self.T_in, D, B, self.dtype)
        self.V = synth.block(seed, layer, "V", 0, B, H_kv, 0, self.T_in, D, B, self.dtype)
        self.q = synth.queries(seed, layer, B, H_q, D, self.dtype)
        self.k_new = new_rows(seed, layer, "K", self.lens_pre, H_kv, D, B, self.dtype)
        self.v_new = new_rows(seed, layer, "V", self.lens_pre, H_kv, D, B, self.dtype)

    def oracle_cache(self, T_max):
        shape = (self.B, self.H_kv, T_max, self.D)
        npdt = np.uint16 if self.dtype == torch.bfloat16 else np.float32
        Kc, Vc = np.zeros(shape, npdt), np.zeros(shape, npdt)
        assert oracle.prefill_write(Kc, Vc, host_bits(self.K), host_bits(self.V), self.lens_pre.numpy()) == 0
        assert oracle.append(Kc, Vc, host_bits(self.k_new), host_bits(self.v_new), self.lens.numpy()) == 0
        return Kc, Vc

    def oracle_out(self, T_max):
        Kc, Vc = self.oracle_cache(T_max)
        return oracle.decode_attn(host_bits(self.q), Kc, Vc, self.lens.numpy())

    def to_device(self, dev="cuda"):
        return {k: getattr(self, k).to(dev) for k in ("K", "V", "q", "k_new", "v_new", "lens_pre", "lens")}


def abs_bits(a: np.ndarray) -> np.ndarray:
    """|x| of an oracle input (bf16 bits or float32)."""
    return (a & 0x7FFF).astype(np.uint16) if a.dtype == np.uint16 else np.abs(a)


def check_close(got: torch.Tensor, ref: np.ndarray, dtype, what="", tight=True, abs_att=None):
    """The tolerance of the decode path: fp32 max abs <= 1e-5; bf16 max abs <= 2e-2 and
    ||got - ref||_2 / ||ref||_2 <= 1e-2.  With `tight` (ref exact, e.g. the oracle's fp64) also:
    every bf16 output within one bf16 ulp of ref, which fp32 accumulation must meet.  The
    tensor-core path rounds each softmax weight to two bf16 terms (16 significant bits, relative
    error <= 2^-16); `abs_att` (the same attention applied to |V|, i.e. sum_t p_t |v_t| / sum_t p_t)
    adds that bound, 2^-16 abs_att, to the one-ulp bar where outputs cancel."""
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    mx = float(err.max()) if err.size else 0.0
    if dtype == torch.float32:
        assert mx <= 1e-5, f"{what}: max abs {mx:.3e}"
        return mx, 0.0
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    assert mx <= 2e-2 and rel <= 1e-2, f"{what}: max abs {mx:.3e} rel {rel:.3e}"
    if not tight:
        return mx, rel
    # one bf16 ulp of the exact value: |ref| = m 2^e with m in [0.5, 1) has ulp 2^(e - 8)
    _, e = np.frexp(np.abs(ref))
    tight = np.ldexp(1.0, e - 8) + 1e-6
    if abs_att is not None:
        tight = tight + 2.0 ** -16 * abs_att
    bad = np.argwhere(err > tight)
    assert bad.size == 0, f"{what}: {len(bad)} outputs beyond one bf16 ulp, first {bad[:3].tolist()}"
    return mx, rel
