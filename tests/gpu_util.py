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


LOG2E = 1.4426950408889634

# Score patterns of ScoreCase, in log2 units (the kernels' domain) along one direction u of
# each KV head: tau(t) for token t.
PATTERNS = {
    "rising": lambda t: 0.05 * t,                       # the maximum moves up every ~160 tokens
    "falling": lambda t: 60.0 - 0.05 * t,               # the maximum first, later scores >= 30 below
    "sawtooth": lambda t: 12.0 * ((t // 97) % 5),       # jumps of 12 > the lazy threshold, mid-tile
}


class ScoreCase:
    """One layer of inputs drawn with torch's CPU generator (fp32 randn, rounded to the cache
    dtype: bf16 round-to-nearest-even), shaped so the online softmax meets what it must handle:
      - "randn": q, K, V ~ N(0, 1);
      - "peaked": q ~ 16 N(0, 1), K, V ~ N(0, 1) (scores of standard deviation ~23 in log2 units);
      - a PATTERNS key: k_t = tau(t) ln2 sqrt(D) u + N(0, 1) and q_j = alpha_j u + 0.3 N(0, 1)
        for a unit vector u per KV head, so query head j sees scores ~ alpha_j tau(t) + noise;
        alpha_j runs from -1.5 to 1.5 over the group (rising and falling histories at once;
        1 for a group of one).
    Same attributes as Case (history of lens_pre[b] tokens, the new token at t = lens_pre[b]),
    with T_q new tokens per sequence when T_q > 1 (q [B, H_q, T_q, D], k_new [B, H_kv, T_q, D])."""

    def __init__(self, kind, seed, B, H_q, H_kv, D, lens_pre, dtype="bf16", T_q=1):
        self.B, self.H_q, self.H_kv, self.D, self.T_q, self.layer = B, H_q, H_kv, D, T_q, 0
        self.dtype = DT[dtype]
        self.lens_pre = torch.as_tensor(lens_pre, dtype=torch.int32)
        self.lens = self.lens_pre + T_q
        G = H_q // H_kv
        T_all = int(self.lens.max())
        g = torch.Generator().manual_seed(seed)
        nk = torch.randn(B, H_kv, T_all, D, generator=g)
        V = torch.randn(B, H_kv, T_all, D, generator=g)
        nq = torch.randn(B, H_q, T_q, D, generator=g)
        if kind == "randn":
            K, q = nk, nq
        elif kind == "peaked":
            K, q = nk, 16.0 * nq
        else:
            u = torch.randn(B, H_kv, 1, D, generator=g)
            u = u / u.norm(dim=-1, keepdim=True)
            t = torch.arange(T_all, dtype=torch.float64).view(1, 1, -1, 1)
            tau = PATTERNS[kind](t).to(torch.float32)
            K = tau * (np.log(2.0) * np.sqrt(D)) * u + nk
            alpha = torch.linspace(-1.5, 1.5, G) if G > 1 else torch.ones(1)
            qd = (alpha.view(1, 1, G, 1, 1) * u.view(B, H_kv, 1, 1, D)).reshape(B, H_q, 1, D)
            q = qd + 0.3 * nq
        K, V, q = K.to(self.dtype), V.to(self.dtype), q.to(self.dtype)
        T_in = max(1, int(self.lens_pre.max()))
        self.K = K[:, :, :T_in].contiguous()
        self.V = V[:, :, :T_in].contiguous()
        lp = [int(x) for x in self.lens_pre]
        kn = torch.stack([K[b, :, lp[b]: lp[b] + T_q] for b in range(B)])
        vn = torch.stack([V[b, :, lp[b]: lp[b] + T_q] for b in range(B)])
        self.k_new = (kn[:, :, 0] if T_q == 1 else kn).contiguous()
        self.v_new = (vn[:, :, 0] if T_q == 1 else vn).contiguous()
        self.q = (q[:, :, 0] if T_q == 1 else q).contiguous()

    oracle_cache = None  # set below (same as Case)

    def to_device(self, dev="cuda"):
        return {k: getattr(self, k).to(dev) for k in ("K", "V", "q", "k_new", "v_new", "lens_pre", "lens")}


class Ref(np.ndarray):
    """An oracle output with `abs_att`, the same attention applied to |V| (None once sliced)."""

    def __array_finalize__(self, obj):
        self.abs_att = None


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
        """The oracle's output, carrying (for check_close) the same attention applied to |V|."""
        Kc, Vc = self.oracle_cache(T_max)
        ref = oracle.decode_attn(host_bits(self.q), Kc, Vc, self.lens.numpy()).view(Ref)
        if self.dtype == torch.bfloat16:
            ref.abs_att = oracle.decode_attn(host_bits(self.q), Kc, np.ascontiguousarray(abs_bits(Vc)),
                                             self.lens.numpy())
        return ref

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
    if abs_att is None:
        abs_att = getattr(ref, "abs_att", None)
    ref = np.asarray(ref)
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


ScoreCase.oracle_cache = Case.oracle_cache
ScoreCase.oracle_out = Case.oracle_out


def abs_att_of(case, Kc, Vc):
    """The oracle's attention applied to |V| (sum_t p_t |v_t| / sum_t p_t): bounds the error the
    kernels' weight rounding can add to an output that cancels (see check_close)."""
    return oracle.decode_attn(host_bits(case.q), Kc, np.ascontiguousarray(abs_bits(Vc)), case.lens.numpy())
