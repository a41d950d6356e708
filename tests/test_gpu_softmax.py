"""GPU parity of the online softmax on inputs that make it work: N(0, 1) data and score
histories whose maximum moves.

The pages define the step as softmax(q K^T / sqrt(D)) V over the whole history ("11.7 KV
Cache：形状、显存与带宽" §2.2; "KV 缓存", "两条数学等价的 decode 路径").  The kernels compute it
in one pass with a running reference maximum that is raised only when a score exceeds it by
a threshold, rescaling the partial sums when it is; the oracle takes the plain two-pass
definition in fp64.  Scores drawn from N(0, 1) data rarely move the maximum after a segment's
first tile, so these cases force it (gpu_util.ScoreCase): peaked attention (q scaled by 16),
rising histories (the maximum is raised many times inside a segment and again after a split
boundary), falling histories (the maximum first, later scores 30+ log2 units below it), and a
sawtooth (jumps above the threshold in the middle of tiles).  Every kernel (CUDA cores, warp
MMA, tcgen05), group sizes 1, 4 and 32 (32: the rescale factors live in shared memory),
several split counts and both merge paths, and one case each of the paged, rolling, several-
new-token and int8 caches.  The bar is the one-bf16-ulp bar of check_close, widened by the
kernels' weight-rounding bound where outputs cancel."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import kvc

from gpu_util import PATTERNS, ScoreCase, abs_att_of, abs_bits, check_close, host_bits

pytestmark = pytest.mark.gpu

KINDS = ["randn", "peaked"] + list(PATTERNS)
LENS = [1500, 3, 700]   # a long stream cut across CTAs, a 4-token one, a middle one
T_MAX = 1600


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()


def _run(case, T_max, math=0, ctas=0, mode=-1, fused=True):
    c = kvc.KVCache(1, case.B, case.H_q, case.H_kv, case.D, T_max, "bf16")
    try:
        c.set_math(math)
        if ctas:
            c.set_ctas(ctas)
        c.set_combine_mode(mode)
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
        return out
    finally:
        c.close()


def _check(case, out, T_max, what):
    Kc, Vc = case.oracle_cache(T_max)
    ref = oracle.decode_attn(host_bits(case.q), Kc, Vc, case.lens.numpy())
    check_close(out, ref, torch.bfloat16, what, abs_att=abs_att_of(case, Kc, Vc))


@pytest.mark.parametrize("math", [1, 2, 3])
@pytest.mark.parametrize("G", [1, 4, 32])
@pytest.mark.parametrize("kind", KINDS)
def test_softmax_patterns_every_kernel(kind, G, math):
    case = ScoreCase(kind, 7000 + 10 * G + math, 3, 2 * G, 2, 128, LENS)
    out = _run(case, T_MAX, math=math, ctas=7)
    _check(case, out, T_MAX, f"{kind} G={G} math={math}")


@pytest.mark.parametrize("math", [1, 3])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("ctas", [1, 7, 152])
@pytest.mark.parametrize("G", [4, 32])
@pytest.mark.parametrize("kind", ["rising", "falling", "sawtooth"])
def test_softmax_patterns_any_split(kind, G, ctas, mode, math):
    case = ScoreCase(kind, 7100 + G + ctas, 3, 2 * G, 2, 128, LENS)
    out = _run(case, T_MAX, math=math, ctas=ctas, mode=mode)
    _check(case, out, T_MAX, f"{kind} G={G} ctas={ctas} mode={mode} math={math}")


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("kind", ["randn", "rising"])
def test_softmax_headline_shape(kind, fused):
    """The 8B-GQA group shape (32 query heads over 8 KV heads) with ragged lengths."""
    case = ScoreCase(kind, 7200, 4, 32, 8, 128, [3000, 17, 2048, 1499])
    out = _run(case, 3100, fused=fused)
    _check(case, out, 3100, f"{kind} 8B-GQA fused={fused}")


@pytest.mark.parametrize("math", [3, 1])
@pytest.mark.parametrize("bs", [16, 128])
def test_softmax_rising_paged(bs, math):
    from test_gpu_paged import _oracle_pool, _run as paged_run, _table
    case = ScoreCase("rising", 7300 + bs, 3, 8, 2, 128, LENS)
    max_blocks = -(-T_MAX // bs)
    table, nbk = _table(7301, LENS, bs, max_blocks)
    out, _, _ = paged_run(case, bs, max_blocks, table, nbk, math=math, ctas=7)
    Kp, Vp = _oracle_pool(case, table, nbk, bs)
    lens = case.lens.numpy()
    ref = oracle.paged_decode_attn(host_bits(case.q), Kp, Vp, table, lens)
    aatt = oracle.paged_decode_attn(host_bits(case.q), Kp, np.ascontiguousarray(abs_bits(Vp)), table, lens)
    check_close(out, ref, torch.bfloat16, f"paged bs={bs} math={math}", abs_att=aatt)


@pytest.mark.parametrize("math", [3, 1])
def test_softmax_sawtooth_rolling(math):
    from test_gpu_rolling import _oracle_ring, _run as rolling_run
    W = 300
    case = ScoreCase("sawtooth", 7400, 3, 8, 2, 128, LENS)
    out, _, _ = rolling_run(case, W, math=math, ctas=7)
    Kr, Vr = _oracle_ring(case, W)
    lens = case.lens.numpy()
    ref = oracle.rolling_decode_attn(host_bits(case.q), Kr, Vr, lens)
    aatt = oracle.rolling_decode_attn(host_bits(case.q), Kr, np.ascontiguousarray(abs_bits(Vr)), lens)
    check_close(out, ref, torch.bfloat16, f"rolling W={W} math={math}", abs_att=aatt)


@pytest.mark.parametrize("math", [3, 1])
@pytest.mark.parametrize("G", [4, 8])
def test_softmax_rising_several_new_tokens(G, math):
    from test_gpu_multi import _run as multi_run
    T_q = 4
    case = ScoreCase("rising", 7500 + G, 3, 2 * G, 2, 128, LENS, T_q=T_q)
    out, _, _ = multi_run(case, T_MAX, math=math, ctas=7)
    npdt = np.uint16
    Kc = np.zeros((case.B, case.H_kv, T_MAX, case.D), npdt)
    Vc = np.zeros_like(Kc)
    assert oracle.prefill_write(Kc, Vc, host_bits(case.K), host_bits(case.V), case.lens_pre.numpy()) == 0
    assert oracle.append_multi(Kc, Vc, host_bits(case.k_new), host_bits(case.v_new), case.lens.numpy()) == 0
    ref = oracle.decode_multi(host_bits(case.q), Kc, Vc, case.lens.numpy())
    aatt = oracle.decode_multi(host_bits(case.q), Kc, np.ascontiguousarray(abs_bits(Vc)), case.lens.numpy())
    check_close(out, ref, torch.bfloat16, f"T_q={T_q} G={G} math={math}", abs_att=aatt)


@pytest.mark.parametrize("G", [4, 8])
@pytest.mark.parametrize("kind", ["rising", "peaked"])
def test_softmax_int8_cache(kind, G):
    from test_gpu_quant import _abs_att, _oracle, _run as quant_run
    case = ScoreCase(kind, 7600 + G, 3, 2 * G, 2, 128, LENS)
    out, _ = quant_run(case, T_MAX, ctas=7)
    qc = _oracle(case, T_MAX)
    ref = qc.decode_attn(host_bits(case.q), case.lens.numpy())
    check_close(out, ref, torch.bfloat16, f"int8 {kind} G={G}", abs_att=_abs_att(case, qc))
