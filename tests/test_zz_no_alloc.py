"""kvc_decode_attn_noalloc: decode attention for callers that cannot allocate device memory.

Such callers (a plugin whose engine owns all device memory, a loop where the allocator's
implicit synchronisation is not allowed) keep the cache in their own buffers and get the
scratch from a fixed array inside the library.  This checks, through the C ABI, that its output
matches the handle-based kvc_decode_attn on the same cache, within the parity tests' tolerance,
on two calls in a row (the shared scratch must be reusable), and that oversized shapes are
refused before anything runs.  The file is named so pytest collects it last."""
import pytest
import torch

from kv_cache_decode_kvc_gb300 import kvc

from gpu_util import Case, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _handle_reference(case, T_max):
    """Cache filled and decoded through the handle API; returns (cache, out)."""
    c = kvc.KVCache(1, case.B, case.H_q, case.H_kv, case.D, T_max,
                    "bf16" if case.dtype == torch.bfloat16 else "f32")
    d = case.to_device()
    c.prefill_write(0, d["K"], d["V"], d["lens_pre"])
    c.append(0, d["k_new"], d["v_new"], d["lens"])
    out = torch.empty(case.B, case.H_q, case.D, dtype=case.dtype, device="cuda")
    c.decode_attn(0, d["q"], out, d["lens"])
    assert c.last_error() == (kvc.KVC_OK, 0)
    return c, d, out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_handle_path_twice(dtype):
    T_max = 3100
    cases = [Case(801, 5, 32, 8, 128, [3000, 17, 2048, 0, 1500], dtype),
             Case(802, 2, 16, 4, 128, [3099, 700], dtype)]
    code = kvc.KVC_BF16 if dtype == "bf16" else kvc.KVC_F32
    for case in cases:  # two calls in a row through the shared scratch
        c, d, ref = _handle_reference(case, T_max)
        try:
            K, V = c.layer_views(0)
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            out = torch.full_like(ref, float("nan"))
            kvc.kvc_decode_attn_noalloc(K, V, case.B, case.H_q, case.H_kv, case.D, T_max, code,
                                        d["q"], out, d["lens"], err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            # both outputs are rounded results, so compare with the tolerance itself (the
            # one-ulp-of-exact bar applies to comparisons against the oracle)
            check_close(out, ref.double().cpu().numpy(), case.dtype, f"noalloc {dtype} B={case.B}",
                        tight=False)
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
