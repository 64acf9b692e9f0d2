"""Host-side checks of the C ABI: the library builds, loads, exports every
symbol include/fl_int4g.h declares, and rejects bad arguments before
launching anything.  No GPU needed (no compute calls)."""
import ctypes
import os
import re

import pytest

import int4_group_quantized_int4g_gb300 as fl
from int4_group_quantized_int4g_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fl_int4g.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return fl.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fl_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(fl.SIGNATURES), set(names) ^ set(fl.SIGNATURES)


def test_status_strings_and_version(L):
    for code in range(8):
        assert isinstance(fl.fl_strerror(code), str) and fl.fl_strerror(code)
    assert fl.fl_strerror(0) == "ok"
    assert fl.fl_int4g_version() >= 100


def test_repacked_bytes(L):
    assert fl.fl_int4g_repacked_bytes(4096, 11008) == 32 * 86 * 8512
    assert fl.fl_int4g_repacked_bytes(200, 384) == 2 * 3 * 8512     # padded to 2 row tiles
    out = ctypes.c_size_t(0)
    assert L.fl_int4g_repacked_bytes(128, 100, 128, ctypes.byref(out)) == 1      # K % 128
    assert L.fl_int4g_repacked_bytes(128, 256, 32, ctypes.byref(out)) == 3       # group 32
    # groups of 64: the super-blocks plus a 320-byte side entry each
    assert fl.fl_int4g_repacked_bytes(200, 384, 64) == 2 * 3 * (8512 + 320)
    assert L.fl_int4g_repacked_bytes(128, 192, 64, ctypes.byref(out)) == 1       # K % 128
    assert L.fl_int4g_repacked_bytes(0, 256, 128, ctypes.byref(out)) == 1
    # groups of 256: the same 128-column super-blocks (two per group)
    assert fl.fl_int4g_repacked_bytes(4096, 11008, 256) == 32 * 86 * 8512
    assert L.fl_int4g_repacked_bytes(128, 384, 256, ctypes.byref(out)) == 1      # K % 256
    assert L.fl_int4g_repacked_bytes(128, 512, 512, ctypes.byref(out)) == 3      # group 512


def test_argument_errors_are_caught_on_the_host(L):
    size = ctypes.c_size_t(0)
    assert L.fl_int4g_linear_workspace(1, 4096, 4096, ctypes.byref(size)) == 0 and size.value > 0
    assert L.fl_int4g_linear_workspace(1, 4096, 4000, ctypes.byref(size)) == 1
    fake = ctypes.c_void_p(0x10000)      # aligned, never dereferenced on the host
    odd = ctypes.c_void_p(0x10008)
    null = None
    # null and misaligned pointers, bad K
    assert L.fl_int4g_linear(null, 1, 256, fake, 128, fake, fake, 1 << 20, None) == 1
    assert L.fl_int4g_linear(odd, 1, 256, fake, 128, fake, fake, 1 << 20, None) == 1
    assert L.fl_int4g_linear(fake, 1, 200, fake, 128, fake, fake, 1 << 20, None) == 1
    assert L.fl_int4g_linear(fake, 0, 256, fake, 128, fake, fake, 1 << 20, None) == 1
    # workspace too small
    assert L.fl_int4g_linear(fake, 1, 256, fake, 128, fake, fake, 16, None) == 2
    assert L.fl_int4g_repack(fake, fake, fake, 128, 256, 128, fake, 100, None) == 1
    assert L.fl_int4g_repack(fake, fake, fake, 128, 256, 32, fake, 1 << 20, None) == 3
    assert L.fl_int4g_repack(fake, fake, fake, 128, 384, 256, fake, 1 << 20, None) == 1
    assert L.fl_int4g_unrepack(fake, 1 << 20, 128, 384, 256, fake, fake, fake, None) == 1
    assert L.fl_int4g_quantize(fake, 128, 384, 256, fake, fake, fake, fake, None) == 1
    assert L.fl_int4g_quantize(fake, 128, 256, 128, fake, fake, null, fake, None) == 1
    assert L.fl_int4g_status(null, None, ctypes.byref(ctypes.c_int())) == 1

    # routing options of fl_moe_int4g_ex, rejected before any launch
    def moe_ex(E, k, scoring, bias, n_group, topk_group, scale):
        r = fl.FlMoeRouting(scoring, 1, bias, n_group, topk_group, scale)
        return L.fl_moe_int4g_ex(fake, fake, 4, 256, E, k, 128, ctypes.byref(r), fake, fake, None, None, fake,
                                 None, None, None, None, fake, 1 << 30, None)
    assert moe_ex(8, 2, fl.FL_SOFTMAX, 0x20000, 1, 1, 1.0) == 1      # a bias needs sigmoid scoring
    assert moe_ex(8, 2, fl.FL_SOFTMAX, None, 4, 2, 1.0) == 1         # so do groups
    assert moe_ex(8, 2, fl.FL_SIGMOID, None, 3, 1, 1.0) == 1         # E % n_group
    assert moe_ex(8, 3, fl.FL_SIGMOID, None, 4, 1, 1.0) == 1         # k > topk_group * E / n_group
    assert moe_ex(8, 2, fl.FL_SIGMOID, None, 4, 5, 1.0) == 1         # topk_group > n_group
    assert moe_ex(8, 2, fl.FL_SIGMOID, 0x20004, 1, 1, 1.0) == 1      # misaligned bias
    assert moe_ex(8, 2, fl.FL_SIGMOID, None, 1, 1, 0.0) == 1         # routed_scale must be positive
    assert moe_ex(8, 2, fl.FL_SIGMOID, None, 1, 1, float("inf")) == 1


def test_decode_plan_fits_shared_memory(L):
    """The decode kernel's plans (host arithmetic, no GPU) over a sweep of
    shapes.  Every plan fits the 227 KB launch limit, or has shed its ring to
    two stages (the launchers then refuse it); the two-per-SM build (M <= 8)
    fits two CTAs per SM; an x region appears only in cluster mode with one
    token tile and at least three stages, its token rows an odd multiple of
    64 bytes apart (conflict-free B-fragment loads), long enough for a rank's
    groups and placed between the zero row and the reduction buffer."""
    KB = 1024
    n = 0
    for M in (1, 2, 5, 8, 9, 16, 17, 32):
        for K in (128, 384, 1024, 4096, 7168, 11008, 16384, 28672, 65536):
            for N in (1, 200, 1024, 3072, 4096, 7168, 11008, 12288, 14336, 32000, 152064):
                for group in (128, 64):
                    for glu in ((0, 1) if M <= 8 else (0,)):
                        for minb in ((0, 3) if M <= 8 else (0,)):
                            for max_cs in (8, 2, 1):
                                p = fl.fl_int4g_test_decode_plan(M, N, K, 152, group, glu, minb, max_cs)
                                if p is None:
                                    assert glu, (M, N, K, group, minb, max_cs)   # only the GLU half declines
                                    continue
                                n += 1
                                where = (M, N, K, group, glu, minb, max_cs, p)
                                assert p["stage_bytes"] % 128 == 0 and p["stages"] >= 2, where
                                assert p["smem"] <= 227 * KB or p["stages"] == 2, where
                                if M <= 8 and minb == 0:
                                    assert p["smem"] <= 113 * KB, where
                                assert p["stages"] * (p["stage_bytes"] + 16) <= p["zrow_off"], where
                                assert p["red_off"] <= p["smem"], where
                                if p["xr_stride"] > 0:
                                    assert M <= 8 and p["csize"] > 1 and p["stages"] >= 3, where
                                    assert p["xr_stride"] % 128 == 64, where
                                    assert p["xr_stride"] >= -(-p["G"] // p["csize"]) * 256, where
                                    assert p["xr_off"] % 128 == 0 and p["xr_off"] >= p["zrow_off"] + 256, where
                                    assert p["xr_off"] + M * p["xr_stride"] <= p["red_off"], where
    assert n > 3000


def test_decode_plan_x_region_choice(L):
    """The Llama- and Qwen-shaped decode linears and the Llama MLP block's
    gate/up half take the x region at every M <= 8; the long-K shapes of the
    GPU parity tests take it at M=1 and fall back to x in the stages at M=8."""
    for M in range(1, 9):
        for K, N, max_cs in ((4096, 12288, 2), (4096, 11008, 8), (11008, 4096, 8), (4096, 4096, 8), (1024, 3072, 8)):
            assert fl.fl_int4g_test_decode_plan(M, N, K, 152, max_cs=max_cs)["xr_stride"] > 0, (M, K, N)
        assert fl.fl_int4g_test_decode_plan(M, 11008, 4096, 152, glu=True)["xr_stride"] > 0, M
    for glu, K, N in ((False, 32768, 1024), (True, 16384, 256)):
        assert fl.fl_int4g_test_decode_plan(1, N, K, 152, glu=glu)["xr_stride"] > 0
        assert fl.fl_int4g_test_decode_plan(8, N, K, 152, glu=glu)["xr_stride"] == 0
    # stream-K (many row tiles) keeps x in the stages
    assert fl.fl_int4g_test_decode_plan(1, 32000, 4096, 152)["csize"] == 1
    assert fl.fl_int4g_test_decode_plan(1, 32000, 4096, 152)["xr_stride"] == 0
    assert fl.fl_int4g_test_decode_plan(1, 0, 4096, 152) is None


def test_decode_plan_sheds_stages_to_fit(L):
    """Groups of 64 at M=32, K=28672, N=7168 (the GPU parity case): the ring
    is cut to fit the 227 KB launch limit, one stage short of overflowing."""
    p = fl.fl_int4g_test_decode_plan(32, 7168, 28672, 152, group=64)
    assert p["smem"] <= 227 * 1024 < p["smem"] + p["stage_bytes"] + 16
    assert p["stages"] > 2
