"""CPU-side checks of the C ABI: the library loads, exports every declared symbol, and its
host-only arithmetic (capacity closed form, split-T partition) is right.  No GPU calls."""
import os
import random

import pytest

from kv_cache_decode_kvc_gb300 import kvc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lib():
    from kv_cache_decode_kvc_gb300 import build
    build.build()
    return kvc.load()


def test_exports_every_header_symbol(lib):
    names = kvc.header_symbols()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def _golden_capacity():
    for line in open(os.path.join(GOLDEN, "capacity.txt"), encoding="utf-8"):
        if line.strip() and not line.startswith("#"):
            name, dims, expected, kind, src = [c.strip() for c in line.split("|")]
            yield name, [int(x) for x in dims.split()], float(expected), kind


@pytest.mark.parametrize("name,dims,expected,kind", list(_golden_capacity()))
def test_bytes_formula_matches_the_pages(lib, name, dims, expected, kind):
    got = kvc.kvc_bytes_formula(*dims)
    if kind == "exact":
        assert got == int(expected), name
    elif kind == "GiB~":
        assert round(got / 2**30) == int(expected), name
    else:
        assert f"{got / 2**20:.3f}" == f"{expected:.3f}", name


def test_bytes_formula_rejects_overflow_and_negatives(lib):
    assert kvc.kvc_bytes_formula(-1, 1, 1, 1, 1, 2) == 0
    assert kvc.kvc_bytes_formula(2**40, 2**40, 1, 1, 1, 2) == 0


def test_partition_covers_every_unit_once(lib):
    rng = random.Random(5)
    for _ in range(200):
        U = rng.randint(1, 10**7)
        P = rng.randint(1, 600)
        # CTA i owns units [floor(i U / P), floor((i+1) U / P)); owner of x is recovered exactly
        for i in rng.sample(range(P), min(P, 8)):
            a, b = i * U // P, (i + 1) * U // P
            for x in {a, b - 1, (a + b) // 2}:
                if a <= x < b:
                    assert kvc.kvc_plan_cta_of(x, U, P) == i
        assert kvc.kvc_plan_cta_of(0, U, P) == 0 or (U * 1) // P == 0
        assert kvc.kvc_plan_cta_of(U - 1, U, P) == P - 1
    assert kvc.kvc_plan_cta_of(5, 5, 3) == -1


def test_split_slots_are_unique(lib):
    # the kernel writes the partial state of (CTA i, stream u) to slot i + u: injective over
    # the pairs whose unit ranges meet (checked by brute force on ragged stream lengths)
    rng = random.Random(9)
    for _ in range(50):
        lens = [rng.randint(0, 700) for _ in range(rng.randint(1, 12))]
        H = rng.randint(1, 4)
        units = [-(-L // 128) for L in lens for _ in range(H)]
        U = sum(units)
        if U == 0:
            continue
        P = rng.randint(1, 40)
        seen = {}
        start = 0
        for u, n in enumerate(units):
            if n:
                for i in range(kvc.kvc_plan_cta_of(start, U, P), kvc.kvc_plan_cta_of(start + n - 1, U, P) + 1):
                    assert (i + u) not in seen, (seen[(i + u)], (i, u))
                    seen[i + u] = (i, u)
            start += n


def test_status_strings(lib):
    assert lib.kvc_status_str(0) == b"ok"
    assert lib.kvc_status_str(kvc.KVC_EUNSUPPORTED) == b"unsupported shape or device"


@pytest.mark.parametrize("args,status", [
    ((1, 2, 6, 4, 128, 16, 0), kvc.KVC_EINVAL),        # H_q % H_kv != 0
    ((0, 2, 8, 4, 128, 16, 0), kvc.KVC_EINVAL),        # no layers
    ((1, 2, 8, 4, 128, 0, 0), kvc.KVC_EINVAL),         # T_max = 0
    ((1, 2, 8, 4, 128, 16, 7), kvc.KVC_EINVAL),        # bad dtype
    ((1, 2048, 8, 4, 128, 16, 0), kvc.KVC_ERANGE),     # B above 1024
    ((1, 2, 8, 4, 96, 16, 0), kvc.KVC_EUNSUPPORTED),   # D not built
    ((1, 2, 4, 4, 4, 16, 0), kvc.KVC_EUNSUPPORTED),    # D = 4 only for fp32
    ((1, 2, 64, 1, 128, 16, 0), kvc.KVC_EUNSUPPORTED), # group of 64
])
def test_create_rejects_bad_shapes_before_touching_the_device(lib, args, status):
    import ctypes
    h = ctypes.c_void_p(123)
    assert lib.kvc_create(ctypes.byref(h), *args) == status
    assert h.value is None


def test_null_handle_calls_are_rejected(lib):
    assert lib.kvc_decode_attn(None, 0, 1, 1, 1, None) == kvc.KVC_EINVAL
    assert lib.kvc_append(None, 0, 1, 1, 1, None) == kvc.KVC_EINVAL
    assert lib.kvc_decode_step(None, 0, 1, 1, 1, 1, 1, None) == kvc.KVC_EINVAL
    assert lib.kvc_prefill_write(None, 0, 1, 1, 1, 1, None) == kvc.KVC_EINVAL
    assert lib.kvc_bytes(None) == 0
    assert lib.kvc_destroy(None) == kvc.KVC_OK


def test_null_handle_setters_are_rejected(lib):
    assert lib.kvc_set_launch_overlap(None, 1) == kvc.KVC_EINVAL
    assert lib.kvc_get_launch_overlap(None) == -1
    assert lib.kvc_set_math(None, 0) == kvc.KVC_EINVAL
    assert lib.kvc_get_math(None) == -1
    assert lib.kvc_set_combine_mode(None, 0) == kvc.KVC_EINVAL


@pytest.mark.parametrize("bad", ["K", "V", "q", "out", "lens", "err"])
def test_noalloc_refuses_misaligned_pointers_before_any_launch(lib, bad):
    # fake device addresses: every check runs on the host, before the device is touched, so a
    # misaligned pointer is refused on a machine without a GPU as well
    ptrs = {"K": 0x10000, "V": 0x20000, "q": 0x30000, "out": 0x40000, "lens": 0x50000, "err": 0x60000}
    ptrs[bad] += 8 if bad in ("K", "V", "q", "out") else 2
    st = lib.kvc_decode_attn_noalloc(ptrs["K"], ptrs["V"], 2, 8, 2, 128, 64, kvc.KVC_BF16, ptrs["q"],
                                     ptrs["out"], ptrs["lens"], ptrs["err"], None)
    assert st == kvc.KVC_EINVAL


def test_wait_selftest_rejects_bad_arguments_on_the_host(lib):
    assert lib.kvc_selftest_wait_timeout(None, 0x1000, 1000, None) == kvc.KVC_EINVAL
    assert lib.kvc_selftest_wait_timeout(0x1000, 0x2004, 1000, None) == kvc.KVC_EINVAL  # info misaligned
    assert lib.kvc_selftest_wait_timeout(0x1000, 0x2000, 3_000_000_000, None) == kvc.KVC_ERANGE
