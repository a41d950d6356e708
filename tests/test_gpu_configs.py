"""Full-size workloads in the launch configuration the benchmark times (fused decode step,
default split), checked against the oracle on sampled sequences: the oracle recomputes
each sampled (sequence, KV head group) from the generator's rows, one by one."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import kvc, synth
from kv_cache_decode_kvc_gb300.workloads import WORKLOADS, fill_layer, step_inputs

from gpu_util import check_close, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _oracle_rows(w, layer, b, lens):
    """Oracle output [H_q, D] of sequence b: its streams are the generator's rows [0, L_b)."""
    L = int(lens[b])
    dt = torch.bfloat16
    K = synth.block(w.seed, layer, "K", b, b + 1, w.H_kv, 0, L, w.D, w.B, dt)
    V = synth.block(w.seed, layer, "V", b, b + 1, w.H_kv, 0, L, w.D, w.B, dt)
    q = synth.queries(w.seed, layer, w.B, w.H_q, w.D, dt)[b : b + 1]
    return oracle.decode_attn(host_bits(q), host_bits(K), host_bits(V), np.array([L], np.int32))[0]


CASES = [
    # workload, layers to run (first and last), sampled sequences
    ("llama2_7b_mha_b1_t4096", [0, 31], [0]),
    ("gqa8b_b24_ragged3000_6000", [0, 31], [0, 7, 13, 23]),
    ("gqa70b_b32_t8192", [0, 79], [0, 19, 31]),
    ("mqa_b64_t4096", [0], [0, 33, 63]),
    ("mqa_b1_t131072", [0], [0]),
]


@pytest.mark.parametrize("name,layers,samples", CASES, ids=[c[0] for c in CASES])
def test_full_size_workload(name, layers, samples):
    w = WORKLOADS[name]
    free, _ = torch.cuda.mem_get_info()
    need = kvc.kvc_bytes_formula(w.layers, w.B, w.H_kv, w.D, w.T_max(), w.elem_bytes)
    if need + (4 << 30) > free:
        pytest.skip(f"needs {need / 2**30:.1f} GiB + 4 GiB margin, {free / 2**30:.1f} GiB free")
    lens = w.lens()
    c = kvc.KVCache(w.layers, w.B, w.H_q, w.H_kv, w.D, w.T_max(), w.dtype)
    try:
        assert c.nbytes() == need
        ld = lens.cuda()
        for layer in layers:
            fill_layer(c, layer, w)
            q, kn, vn = step_inputs(w, layer)
            out = torch.empty(w.B, w.H_q, w.D, dtype=torch.bfloat16, device="cuda")
            c.decode_step(layer, q, kn, vn, out, ld)
            assert c.last_error() == (kvc.KVC_OK, 0)
            for b in samples:
                ref = _oracle_rows(w, layer, b, lens)
                check_close(out[b], ref, torch.bfloat16, f"{name} layer {layer} b {b}")
            # the append wrote the generator's row T_b into slot T_b, bit for bit
            Kv, Vv = c.layer_views(layer)
            for b in samples:
                L = int(lens[b])
                assert torch.equal(Kv[b, :, L - 1], kn[b]) and torch.equal(Vv[b, :, L - 1], vn[b])
            del q, kn, vn, out
    finally:
        c.close()
        torch.cuda.empty_cache()
