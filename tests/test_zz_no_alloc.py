"""kvc_decode_attn_noalloc: decode attention for callers that cannot allocate device memory.

Such callers (a plugin whose engine owns all device memory, a loop where the allocator's
implicit synchronisation is not allowed) keep the cache in their own buffers and get the
scratch from a fixed array inside the library.  Through the C ABI, this checks that its output
matches the oracle at the parity tests' one-ulp bar and the handle-based kvc_decode_attn within
the tolerance, on two calls in a row (the shared scratch must be reusable); that a split-T
shape merged by the separate combine kernel works from the scratch too; that bad lengths reach
the caller's error word; that no device memory is taken; and that oversized shapes are refused
before anything runs.  The file is named so pytest collects it last."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_decode_kvc_gb300 import kvc

from gpu_util import Case, abs_att_of, check_close, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _handle_reference(case, T_max):
    """Cache filled and decoded through the handle API; returns (cache, device inputs, out)."""
    c = kvc.KVCache(1, case.B, case.H_q, case.H_kv, case.D, T_max,
                    "bf16" if case.dtype == torch.bfloat16 else "f32")
    d = case.to_device()
    c.prefill_write(0, d["K"], d["V"], d["lens_pre"])
    c.append(0, d["k_new"], d["v_new"], d["lens"])
    out = torch.empty(case.B, case.H_q, case.D, dtype=case.dtype, device="cuda")
    c.decode_attn(0, d["q"], out, d["lens"])
    assert c.last_error() == (kvc.KVC_OK, 0)
    return c, d, out


def _noalloc(c, case, T_max, d, lens=None):
    K, V = c.layer_views(0)
    code = kvc.KVC_BF16 if case.dtype == torch.bfloat16 else kvc.KVC_F32
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((case.B, case.H_q, case.D), float("nan"), dtype=case.dtype, device="cuda")
    kvc.kvc_decode_attn_noalloc(K, V, case.B, case.H_q, case.H_kv, case.D, T_max, code,
                                d["q"], out, d["lens"] if lens is None else lens, err)
    torch.cuda.synchronize()
    return out, int(err.item())


def _oracle_check(case, T_max, out, what):
    Kc, Vc = case.oracle_cache(T_max)
    ref = oracle.decode_attn(host_bits(case.q), Kc, Vc, case.lens.numpy())
    aatt = abs_att_of(case, Kc, Vc) if case.dtype == torch.bfloat16 else None
    check_close(out, ref, case.dtype, what, abs_att=aatt)


# (seed, B, H_q, H_kv, lens_pre): GQA with ragged lengths (merged by the last CTA of a stream);
# MQA with one long stream (merged by the separate combine kernel, from the scratch array)
SHAPES = [(801, 5, 32, 8, [3000, 17, 2048, 0, 1500]),
          (802, 2, 16, 4, [3099, 700]),
          (803, 1, 32, 1, [3099])]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_oracle_and_handle_path_twice(dtype):
    T_max = 3100
    for seed, B, H_q, H_kv, lp in SHAPES:  # calls in a row through the shared scratch
        case = Case(seed, B, H_q, H_kv, 128, lp, dtype)
        c, d, ref = _handle_reference(case, T_max)
        try:
            for rep in range(2):
                out, err = _noalloc(c, case, T_max, d)
                assert err == 0
                _oracle_check(case, T_max, out, f"noalloc {dtype} B={B} G={H_q // H_kv} call {rep}")
                # both are rounded results: the handle path is compared within the tolerance
                check_close(out, ref.double().cpu().numpy(), case.dtype, f"noalloc vs handle {dtype}",
                            tight=False)
        finally:
            c.close()


def test_noalloc_takes_no_device_memory():
    case = Case(804, 3, 32, 1, 128, [2000, 5, 999], "bf16")
    T_max = 2048
    c, d, _ = _handle_reference(case, T_max)
    try:
        _noalloc(c, case, T_max, d)  # first call on the device: scratch address, kernels loaded
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        out, err = _noalloc(c, case, T_max, d)
        out2, err2 = _noalloc(c, case, T_max, d)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert err == 0 and err2 == 0
        _oracle_check(case, T_max, out2, "noalloc after the memory check")
    finally:
        c.close()


def test_noalloc_reports_bad_lengths_in_err():
    case = Case(805, 3, 8, 2, 128, [10, 20, 30], "bf16")
    T_max = 64
    c, d, _ = _handle_reference(case, T_max)
    try:
        bad = torch.tensor([11, 0, T_max + 3], dtype=torch.int32, device="cuda")
        out, err = _noalloc(c, case, T_max, d, lens=bad)
        assert err & kvc.KVC_DEV_BAD_LENS
        assert not out[1].float().abs().sum() and not out[2].float().abs().sum()
        # the valid row is still right; a following good call reports nothing
        Kc, Vc = case.oracle_cache(T_max)
        ref = oracle.decode_attn(host_bits(case.q), Kc, Vc, case.lens.numpy())
        check_close(out[:1], ref[:1], torch.bfloat16, "valid row beside bad ones")
        _, err = _noalloc(c, case, T_max, d)
        assert err == 0
    finally:
        c.close()


def test_noalloc_refuses_shapes_beyond_its_scratch():
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1024, dtype=torch.int32, device="cuda")
    with pytest.raises(kvc.KvcError) as ei:
        # 1024 x 32 streams x 32 heads x 256 partial outputs: far beyond the fixed scratch
        kvc.kvc_decode_attn_noalloc(dummy, dummy, 1024, 1024, 32, 256, 8, kvc.KVC_BF16,
                                    dummy, dummy, lens)
    assert ei.value.status == kvc.KVC_ERANGE
