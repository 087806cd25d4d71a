"""Host-side checks of the C ABI: no GPU needed, nothing is launched.

The library must load, export every function declared in include/dbw_gemm.h,
reject every precondition violation with its status code before touching a
device, and plan launches as a pure function of the sizes and the SM count.
"""
import ctypes
import os
import re
import subprocess

import pytest

from dense_bit_weight_gb300 import build as _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dbw_gemm.h")


@pytest.fixture(scope="module")
def g():
    _build.build()
    from dense_bit_weight_gb300 import gemm
    return gemm


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gemm_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(g):
    names = declared_functions()
    assert {"gemm_bf16", "gemm_w4a16", "gemm_last_device_error", "gemm_status_string",
            "gemm_shutdown"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", g._LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(\w+)$", out, flags=re.M))
    for n in names:
        assert n in exported, n
        assert hasattr(g.lib, n)
    assert sorted(names) == sorted(g.EXPORTS)


def test_status_strings(g):
    for code in range(0, 11):
        s = g.gemm_status_string(code)
        assert s and s != "unknown status"
    assert g.gemm_status_string(99) == "unknown status"


A16 = 1 << 20   # a fake 16-byte aligned address: never dereferenced, nothing launches


def bf16(**kw):
    a = dict(A=A16, B=A16 * 4, C=A16 * 8, M=4, N=16, K=32, lda=32, ldb=32, ldc=16)
    a.update(kw)
    return a


def call_bf16(g, **kw):
    a = bf16(**kw)
    return g.gemm_bf16_ptr(a["A"], a["B"], a["C"], a["M"], a["N"], a["K"], a["lda"], a["ldb"], a["ldc"])


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), 2), (dict(N=-3), 2), (dict(K=-8), 2), (dict(K=12, lda=16, ldb=16), 2),
    (dict(K=1 << 31, lda=1 << 31, ldb=1 << 31), 2),
    (dict(A=0), 1), (dict(B=0), 1), (dict(C=0), 1),
    (dict(lda=24), 3), (dict(ldb=36), 3), (dict(ldc=8), 3), (dict(ldc=20), 3),
    (dict(A=A16 + 2), 4), (dict(B=A16 * 4 + 8), 4), (dict(C=A16 * 8 + 4), 4),
    (dict(C=A16 + 64), 9), (dict(C=A16 * 4), 9),
])
def test_bf16_rejects_before_launch(g, kw, code):
    assert call_bf16(g, **kw) == code


def test_bf16_empty_is_ok_without_device(g):
    # M == 0 or N == 0: nothing to do, no device needed
    assert call_bf16(g, M=0) == 0
    assert call_bf16(g, N=0, ldc=8) == 0
    assert call_bf16(g, M=0, A=0, B=0) == 0


def call_w4(g, **kw):
    a = dict(A=A16, Bq=A16 * 4, S=A16 * 8, Z=A16 * 12, C=A16 * 16, M=1, N=64, K=256, group=128)
    a.update(kw)
    return g.gemm_w4a16_ptr(a["A"], a["Bq"], a["S"], a["Z"], a["C"], a["M"], a["N"], a["K"], a["group"])


@pytest.mark.parametrize("kw,code", [
    (dict(group=16), 5), (dict(group=96), 5), (dict(K=320, group=128), 5), (dict(group=0), 5),
    (dict(K=0), 2), (dict(N=12), 2), (dict(M=-1), 2),
    (dict(A=0), 1), (dict(Bq=0), 1), (dict(S=0), 1), (dict(Z=0), 1), (dict(C=0), 1),
    (dict(A=A16 + 8), 4), (dict(Bq=A16 * 4 + 4), 4), (dict(C=A16 * 16 + 2), 4), (dict(S=A16 * 8 + 1), 4),
    (dict(C=A16 * 4 + 32), 9),
])
def test_w4a16_rejects_before_launch(g, kw, code):
    assert call_w4(g, **kw) == code


def test_plans_are_host_only_and_cover_the_workloads(g):
    sms = 152
    for M in (1, 8, 32, 128):
        for N, K in ((6144, 4096), (4096, 4096), (24576, 4096)):
            p = g.gemm_bf16_plan(M, N, K, num_sms=sms)
            assert p["variant"] in (1, 2, 3, 10) and p["kernels"] >= 1 and p["grid"] >= 1
    for M in (1024, 4096, 16384):
        p = g.gemm_bf16_plan(M, 8192, 8192, num_sms=sms)
        assert p["variant"] == 9 and p["tile_m"] == p["tile_n"] == 256
    assert g.gemm_bf16_plan(5, 7, 0, num_sms=sms)["variant"] == 4
    for M in (1, 16, 64, 128):
        p = g.gemm_w4a16_plan(M, 7168, 5120, 128, num_sms=sms)
        assert p["variant"] in (1, 2, 3, 5, 6)
    # W4A16: M <= 8 the TMA-fed fragment kernel, 9 <= M <= 128 tcgen05
    for M in (1, 2, 4, 5, 8):
        p = g.gemm_w4a16_plan(M, 34816, 5120, 128, num_sms=sms)
        assert p["variant"] == 6 and p["tile_m"] == 8 and p["kernels"] == 2
    for M in (9, 16, 128, 129, 1023):
        assert g.gemm_w4a16_plan(M, 34816, 5120, 128, num_sms=sms)["variant"] == 2
    # more than 128 tokens on the tcgen05 W4A16 kernel: 128-token tiles
    p = g.gemm_w4a16_plan(1000, 34816, 5120, 128, num_sms=sms)
    assert p["tile_m"] == 128 and p["grid"] <= sms
    # from 1024 tokens, waves of pair tiles at least 3/4 full: weights
    # dequantised once, then the pair GEMM
    for M in (1024, 4096):
        p = g.gemm_w4a16_plan(M, 34816, 5120, 128, num_sms=sms)
        assert (p["variant"], p["kernels"], p["tile_m"]) == (9, 2, 256) and p["grid"] <= sms
    assert g.gemm_w4a16_plan(4096, 5120, 17408, 128, num_sms=sms)["variant"] == 9     # 320 pair tiles: 0.84
    assert g.gemm_w4a16_plan(1024, 5120, 17408, 128, num_sms=sms)["variant"] == 2     # 80 pair tiles: 0.53
    # the one-kernel fragment plan stages a tile's scale rows whole (up to
    # 192 groups); beyond, the pre-pass fragment kernel (scales per stage)
    assert g.gemm_w4a16_plan(1, 4096, 32 * 192, 32, num_sms=sms)["kernels"] == 1
    p = g.gemm_w4a16_plan(1, 4096, 32 * 545, 32, num_sms=sms)
    assert (p["variant"], p["kernels"]) == (6, 2)
    assert g.gemm_w4a16_plan(16, 4096, 32 * 545, 32, num_sms=sms)["variant"] == 2
    # beyond the staged-scale limit (K / group > 544 groups) the register kernel does not plan
    with pytest.raises(g.GemmError):
        g.gemm_w4a16_plan(1, 4096, 32 * 545, 32, "register", num_sms=sms)
    # up to three CTAs per SM: a cluster of two CTAs per 32-row tile, its
    # eight warps sharing the 128-k chunks of K (one kernel); more tiles: the
    # activation pre-pass, then 32-row tiles shared by 1, 2 or 4 warps
    p = g.gemm_w4a16_plan(1, 7168, 5120, 128, num_sms=sms)      # 224 tiles
    assert (p["variant"], p["kernels"], p["grid"], p["split"], p["tile_n"]) == (6, 1, 448, 8, 32)
    p = g.gemm_w4a16_plan(16, 5120, 17408, 128, num_sms=sms)    # M = 16 too
    assert (p["variant"], p["kernels"], p["grid"], p["tile_m"]) == (6, 1, 320, 16)
    p = g.gemm_w4a16_plan(1, 5120, 256, 128, num_sms=sms)       # two chunks: two warps
    assert (p["grid"], p["split"]) == (320, 2)
    p = g.gemm_w4a16_plan(1, 34816, 5120, 128, num_sms=sms)     # 1088 tiles: pre-pass kernel
    assert (p["variant"], p["kernels"], p["split"]) == (6, 2, 2)
    assert g.gemm_w4a16_plan(16, 34816, 5120, 128, num_sms=sms)["variant"] == 2
    with pytest.raises(g.GemmError):
        g.gemm_bf16_plan(4, 4, 4, num_sms=sms)       # K % 8
    with pytest.raises(g.GemmError):
        g.gemm_w4a16_plan(4, 64, 256, 48, num_sms=sms)


def test_binding_fails_loudly_without_library(tmp_path):
    # the binding must raise, not fall back, when the shared library is absent
    code = (
        "import sys, os, importlib.util\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import dense_bit_weight_gb300.gemm as m\n"
        "src = m.__file__\n"
        "spec = importlib.util.spec_from_file_location('g2', src)\n"
        "mod = importlib.util.module_from_spec(spec)\n"
        "m_path = m._LIB_PATH\n"
        "import builtins\n"
        "real = os.path.exists\n"
        "os.path.exists = lambda p: False if p == m_path else real(p)\n"
        "try:\n"
        "    spec.loader.exec_module(mod)\n"
        "except ImportError as e:\n"
        "    print('raised', 'missing' in str(e))\n"
    )
    out = subprocess.run(["python", "-c", code], capture_output=True, text=True)
    assert "raised True" in out.stdout, out.stdout + out.stderr


def test_k_zero_ignores_empty_inputs(g):
    # K == 0: A and B are empty and never read, so their pointers and leading
    # dimensions are not checked (the call still needs a device, so only the
    # C-side checks are observable here)
    assert call_bf16(g, K=0, A=0, B=0, lda=1, ldb=3, ldc=5) == 3      # ldc still checked
    assert call_bf16(g, K=0, A=0, B=0, C=0) == 1


def test_fused_epilogue_argument_errors():
    # rejected before any device work: an unknown epilogue, a bias where none is
    # used, no bias where one is required (GEMM_ERR_EPILOGUE = 11)
    from dense_bit_weight_gb300 import gemm as g
    p = 1 << 20   # never dereferenced
    assert g.gemm_bf16_fused_ptr(p, p, 0, p, 8, 8, 8, 8, 8, 8, 7) == 11
    assert g.gemm_bf16_fused_ptr(p, p, 0, p, 8, 8, 8, 8, 8, 8, 1) == 11
    assert g.gemm_bf16_fused_ptr(p, p, p, p, 8, 8, 8, 8, 8, 8, 2) == 11
    assert g.gemm_bf16_fused_ptr(p, p, p, p, 8, 8, 8, 8, 8, 8, 0) == 11
    for epi in (3, 4, 5):                        # the bias + activation epilogues need a bias
        assert g.gemm_bf16_fused_ptr(p, p, 0, p, 8, 8, 8, 8, 8, 8, epi) == 11
    assert g.gemm_bf16_fused_ptr(p, p, 0, p, 8, 8, 8, 8, 8, 8, -1) == 11
    assert g.gemm_status_string(11) != g.gemm_status_string(99)
    # every fused epilogue runs on CTA pairs at prefill sizes too (256 weight
    # rows per pair tile: 128 output columns for the (gate, up) row pairs)
    for epi in ("bias", "silu_mul", "bias_relu", "bias_silu", "bias_gelu"):
        p = g.gemm_bf16_fused_plan(4096, 8192, 8192, epi, num_sms=152)
        assert (p["variant"], p["tile_m"], p["tile_n"]) == (9, 256, 256)
    # the SiLU-mul plans are plans on the 2N weight rows: single-CTA kernels up
    # to 128 tokens, CTA pairs beyond
    sms = 152
    for M in (1, 8, 128):
        assert g.gemm_bf16_fused_plan(M, 12288, 4096, "silu_mul", num_sms=sms)["variant"] in (1, 2, 3)
    assert g.gemm_bf16_fused_plan(4096, 12288, 4096, "silu_mul", num_sms=sms)["variant"] == 9


def test_prefill_last_wave_split():
    # a last wave a quarter to half full is split along K (2 or 3 CTAs per
    # leftover tile, whole tiles before); a smaller leftover stays whole tiles
    from dense_bit_weight_gb300 import gemm as g
    sms = 152
    pf = lambda M, N, K: g.gemm_bf16_plan(M, N, K, "prefill", num_sms=sms)   # the single-CTA kernel
    assert pf(1024, 6144, 4096)["split"] == 3      # 192 tiles: 152 + 40
    assert pf(4096, 4096, 4096)["split"] == 2      # 512 tiles: 456 + 56
    assert pf(4096, 24576, 4096)["split"] == 1     # 3072 tiles: 3040 + 32


def test_prefill_on_cta_pairs():
    # 256 x 256 pair tiles whenever they keep at least half the SM pairs busy;
    # the grid is two CTAs per pair, at most one pair per two SMs
    from dense_bit_weight_gb300 import gemm as g
    sms = 152
    p = g.gemm_bf16_plan(1024, 4096, 4096, num_sms=sms)          # 4 x 16 = 64 pair tiles
    assert (p["variant"], p["grid"], p["tile_m"], p["tile_n"]) == (9, 128, 256, 256)
    assert g.gemm_bf16_plan(4096, 24576, 4096, num_sms=sms)["grid"] == sms
    assert g.gemm_bf16_plan(512, 4096, 12288, num_sms=sms)["variant"] == 3    # 32 pair tiles: stream-K instead
    assert g.gemm_bf16_plan(300, 1200, 4096, num_sms=sms)["variant"] == 3
    # fused epilogues take the pair kernel too; it can be forced
    assert g.gemm_bf16_fused_plan(4096, 12288, 4096, "silu_mul", num_sms=sms)["variant"] == 9
    assert g.gemm_bf16_plan(8, 64, 64, "pair", num_sms=sms)["grid"] == 2


def test_band_plans():
    # the band kernel: one band of at most 64 weight rows per SM, tokens in
    # MMA tiles of 8 (at most 32); a ring of eight stages (two per MMA warp),
    # or one slot per stage when K spans at most four
    from dense_bit_weight_gb300 import gemm as g
    sms = 152
    plan = lambda M, N, K: g.gemm_bf16_plan(M, N, K, "band", num_sms=sms)
    p = plan(1, 6144, 4096)
    assert (p["variant"], p["grid"], p["tile_m"], p["tile_n"], p["stages"]) == (10, 152, 8, 41, 8)
    p = plan(32, 9728, 520)                                    # 64-row bands, 32 tokens, nine 64-k stages
    assert (p["grid"], p["tile_m"], p["tile_n"], p["stages"]) == (152, 32, 64, 8)
    assert plan(1, 4096, 256)["stages"] == 1                   # K in one stage: one slot
    assert plan(9, 64, 2056)["grid"] == 64                     # one row per CTA
    assert plan(16, 4096, 12288)["tile_m"] == 16
    for M, N in ((33, 4096), (1, 9729)):                       # too many tokens / a band of 65 rows
        with pytest.raises(g.GemmError):
            plan(M, N, 4096)
    # the bias epilogues run on it; the SiLU-mul (gate, up) pairs do not
    assert g.gemm_bf16_fused_plan(8, 4096, 4096, "bias_gelu", "band", num_sms=sms)["variant"] == 10
    with pytest.raises(g.GemmError):
        g.gemm_bf16_fused_plan(8, 4096, 4096, "silu_mul", "band", num_sms=sms)


def test_w4a16_band_plans():
    # the W4A16 band kernel (forced only): up to 8 tokens, bands of at most 48
    # rows, at most 192 quantisation groups per row; a band that fits shared
    # memory whole goes in four stages, a longer one through eight slots
    from dense_bit_weight_gb300 import gemm as g
    plan = lambda M, N, K, grp: g.gemm_w4a16_plan(M, N, K, grp, "band", num_sms=152)
    p = plan(1, 7168, 5120, 128)
    assert (p["variant"], p["grid"], p["tile_m"], p["tile_n"], p["stages"]) == (10, 152, 8, 48, 4)
    assert plan(8, 5120, 17408, 128)["stages"] == 8
    for args in ((9, 7168, 5120, 128), (1, 7304, 5120, 128), (1, 5120, 17408, 32)):
        with pytest.raises(g.GemmError):
            plan(*args)
    assert g.gemm_w4a16_plan(1, 7168, 5120, 128, num_sms=152)["variant_name"] == "fragment"   # not routed


def test_pair_schedules():
    # whole pair tiles round-robin when they fill at least half the pairs;
    # a last wave of a quarter to half the pairs: full waves whole, each
    # leftover tile split along K among up to three pairs; fewer tiles:
    # stream-K over the largest multiple of the token tile-rows that fits the
    # pairs (the tile-rows then run in lockstep)
    from dense_bit_weight_gb300 import gemm as g
    sms = 152
    plan = lambda M, N, K: g.gemm_bf16_plan(M, N, K, "pair", num_sms=sms)
    assert (plan(1024, 4096, 4096)["split"], plan(1024, 4096, 4096)["grid"]) == (1, 128)   # 64 tiles
    # a leftover quarter to half wave is split along K only on a long K
    # (the fixup costs about 48 k-blocks)
    assert (plan(1024, 6144, 4096)["split"], plan(1024, 6144, 4096)["grid"]) == (1, 152)   # 96: 76 + 20, 64 k-blocks
    assert (plan(768, 8192, 8192)["split"], plan(768, 8192, 8192)["grid"]) == (3, 152)     # 96, 128 k-blocks
    assert plan(4096, 4096, 4096)["split"] == 1                                            # 256: 228 + 28
    assert plan(4096, 4096, 12288)["split"] == 2                                           # 192 k-blocks
    assert plan(4096, 24576, 4096)["split"] == 1                                           # 1536: 1520 + 16
    assert plan(4096, 6144, 4096)["split"] == 1                                            # 384: 380 + 4
    p = plan(512, 4096, 12288)                                                             # 32 tiles
    assert p["grid"] == sms and p["split"] >= 2
    p = plan(700, 1000, 1000)                                                              # 12 tiles x 16 k-blocks
    assert p["grid"] == 2 * (76 // 3 * 3) and p["split"] >= 2                              # 3 tile-rows: 75 pairs
    assert plan(300, 4096, 12288)["grid"] == 2 * 76                                        # 2 tile-rows
    assert plan(256, 4096, 12288)["grid"] == 2 * 76                                        # one tile-row
    assert plan(129, 4104, 8)["split"] == 1                                                # 17 units: too few to share


def test_single_cta_stream_k_grid_is_a_multiple_of_the_token_tiles():
    # single-CTA prefill under stream-K: the grid is the largest multiple of
    # the 128-row token tiles within the SMs
    from dense_bit_weight_gb300 import gemm as g
    sms = 152
    plan = lambda M, N, K: g.gemm_bf16_plan(M, N, K, "prefill", num_sms=sms)
    assert plan(512, 4096, 12288)["grid"] == 152                                           # 4 tile-rows
    assert plan(384, 4096, 12288)["grid"] == 150                                           # 3 tile-rows
    assert plan(640, 2048, 12288)["grid"] == 150                                           # 5 tile-rows x 8
    assert plan(128, 4096, 12288)["grid"] == 152                                           # 1 tile-row


def test_wide_tiles_for_one_token_tile():
    # M <= 128 and a weight count that fills one wave of 176-256-row tiles:
    # the prefill kernel, weights read once each; otherwise the skinny split-K
    from dense_bit_weight_gb300 import gemm as g
    sms = 152
    for M in (1, 4, 5, 8, 16, 32, 128):
        p = g.gemm_bf16_plan(M, 24576, 4096, num_sms=sms)
        assert (p["variant"], p["tile_n"], p["grid"], p["split"]) == (3, 176, 140, 1)
    assert g.gemm_bf16_plan(64, 28000, 4096, num_sms=sms)["tile_n"] == 192      # 146 tiles
    assert g.gemm_bf16_plan(64, 32768, 4096, num_sms=sms)["tile_n"] == 224      # 147 tiles
    assert g.gemm_bf16_plan(128, 16384, 4096, num_sms=sms)["variant"] == 2      # 176 rows: 94 tiles, too few
    assert g.gemm_bf16_plan(128, 4096, 4096, num_sms=sms)["variant"] == 2
    assert g.gemm_bf16_plan(129, 24576, 4096, num_sms=sms)["tile_n"] == 256     # two token tiles
    assert g.gemm_bf16_plan(4, 4096, 4096, num_sms=sms)["variant"] == 10        # band kernel at 2-4 tokens
    assert g.gemm_bf16_plan(1, 4096, 4096, num_sms=sms)["variant"] == 1         # GEMV: 1 token, 27-row bands
    assert g.gemm_bf16_plan(1, 6144, 4096, num_sms=sms)["variant"] == 10        # band: 41-row bands
    assert g.gemm_bf16_plan(8, 4096, 12288, num_sms=sms)["variant"] == 2        # skinny beyond K = 8192
    assert g.gemm_bf16_plan(16, 6144, 4096, num_sms=sms)["variant"] == 2        # skinny from 9 tokens
    # forced variants keep their kernels; the fused gate/up pairs take the same tiles
    assert g.gemm_bf16_plan(128, 24576, 4096, "skinny", num_sms=sms)["variant"] == 2
    assert g.gemm_bf16_plan(128, 2 * 12288, 4096, num_sms=sms)["tile_n"] == 176
    # the fused gate/up pairs (C 12288 columns) take them from 64 tokens on
    for M, variant in ((1, 1), (8, 2), (32, 2), (64, 3), (128, 3)):
        assert g.gemm_bf16_fused_plan(M, 12288, 4096, "silu_mul", num_sms=sms)["variant"] == variant
    assert g.gemm_bf16_fused_plan(8, 24576, 4096, "bias", num_sms=sms)["tile_n"] == 176
    assert g.gemm_bf16_fused_plan(8, 24576, 4096, "none", num_sms=sms) == g.gemm_bf16_plan(8, 24576, 4096, num_sms=sms)
    with pytest.raises(g.GemmError):
        g.gemm_bf16_fused_plan(8, 24576, 4096, 7, num_sms=sms)              # unknown epilogue
    with pytest.raises(g.GemmError):
        g.gemm_bf16_fused_plan(8, 2 ** 30 + 8, 4096, "silu_mul", num_sms=sms)  # 2N weight rows too many
    with pytest.raises(g.GemmError):
        g.gemm_bf16_fused_plan(200, 24576, 4096, "silu_mul", "skinny", num_sms=sms)
    with pytest.raises(g.GemmError):
        g.gemm_bf16_fused_plan(8, 24576, 12, "bias", num_sms=sms)            # K % 8
    assert g.gemm_bf16_fused_plan(8, 24576, 4096, "bias", "gemv", num_sms=sms)["variant"] == 1


def test_planner_invariants_over_shapes():
    # every AUTO plan over a spread of decode and prefill shapes is one the
    # kernels accept: a known family, a grid within the SM count (persistent
    # kernels) or a positive GEMV grid, wide weight tiles in one wave filling
    # at least 85% of the SMs, and split plans that leave every CTA work
    from dense_bit_weight_gb300 import gemm as g
    import random
    rnd = random.Random(7)
    for sms in (152, 148, 132):
        for _ in range(400):
            M = rnd.choice([1, 2, 3, 4, 5, 8, 15, 16, 17, 31, 32, 64, 100, 128, 129, 512, 4096])
            N = rnd.randrange(8, 40000, 8)
            K = rnd.randrange(8, 16384, 8)
            p = g.gemm_bf16_plan(M, N, K, num_sms=sms)
            assert p["variant"] in (1, 2, 3, 9, 10), p
            assert p["grid"] >= 1 and p["split"] >= 1
            if p["variant"] == 10:   # band: one band of at most 64 rows per CTA, at most 8 tokens
                assert M <= 8 and p["grid"] == min(N, sms) and p["tile_n"] <= 64 and p["split"] == 1, (M, N, K, p)
            if p["variant"] in (2, 3):
                assert p["grid"] <= 2 * sms, (M, N, K, p)
            if p["variant"] == 9:
                assert M > 128 and p["grid"] % 2 == 0 and p["grid"] <= sms, (M, N, K, p)
            if p["variant"] == 3 and M <= 128 and p["tile_n"] != 256:
                tiles = -(-N // p["tile_n"])
                assert p["tile_n"] in (176, 192, 224) and p["tile_n"] >= M
                assert tiles == p["grid"] and 0.85 * sms <= tiles <= sms, (M, N, K, p)
            if p["variant"] == 2 and -(-N // 128) <= sms:   # one wave of weight tiles: cluster split-K
                assert p["grid"] == -(-N // 128) * p["split"] and p["split"] <= 8 and p["grid"] <= sms


class _FakeCudaTensor:
    """Stands in for a CUDA bf16 tensor (no GPU here): only the attributes the
    binding reads before it reaches the C call."""

    def __init__(self, shape, dtype=None, device_index=0):
        import torch
        self.shape = tuple(shape)
        self.dtype = dtype or torch.bfloat16
        self.is_cuda = True
        self.device = torch.device("cuda", device_index)

    def dim(self):
        return len(self.shape)

    def stride(self, i=None):
        st = (self.shape[1], 1) if len(self.shape) == 2 else (1,)
        return st if i is None else st[i]

    def is_contiguous(self):
        return True

    def data_ptr(self):
        raise AssertionError("the binding must reject the call before reading pointers")


def test_binding_rejects_host_and_cross_device_tensors():
    import torch
    from dense_bit_weight_gb300 import gemm as g
    A, B = _FakeCudaTensor((4, 64)), _FakeCudaTensor((32, 64))
    with pytest.raises(ValueError):
        g.gemm_bf16(A, B, C=torch.empty((4, 32), dtype=torch.bfloat16))            # C in host memory
    with pytest.raises(ValueError):
        g.gemm_bf16(A, _FakeCudaTensor((32, 64), device_index=1), C=_FakeCudaTensor((4, 32)))
    with pytest.raises(ValueError):
        g.gemm_bf16_fused(A, B, bias=torch.zeros(32, dtype=torch.bfloat16), C=_FakeCudaTensor((4, 32)))
    with pytest.raises(ValueError):
        g.gemm_bf16(torch.empty((4, 64), dtype=torch.bfloat16), B)                 # A in host memory


def test_mx_plans_cover_both_schedules(g):
    p = g.gemm_mx_plan(4096, 8192, 1024, num_sms=152)               # 1024 tiles: whole tiles on every SM
    assert p["grid"] == 152 and p["split"] == 1 and p["kernels"] == 2
    p = g.gemm_mx_plan(1024, 1024, 1024, num_sms=152)               # 32 tiles: stream-K over the SMs
    assert p["grid"] == 152 and p["split"] > 1 and p["tile_n"] == 256
    assert g.gemm_mx_plan(37, 120, 384, num_sms=152)["tile_n"] == 128
    assert g.gemm_mx_plan(32, 64, 0, num_sms=152)["variant_name"] == "zero"


def test_mx_rejects_bad_arguments_before_launch(g):
    a = 1 << 20
    assert g.gemm_mx_ptr("e4m3", a, a, a, a, a * 64, 4, 16, 96) == 2          # K % 128
    assert g.gemm_mx_ptr("e4m3", a, a, a, a, a * 64, 4, 12, 128) == 2         # N % 8
    assert g.gemm_mx_ptr("e4m3", a, a, a, a, a * 64, -1, 16, 128) == 2
    assert g.gemm_mx_ptr("e4m3", a + 8, a, a, a, a * 64, 4, 16, 128) == 4     # A alignment
    assert g.gemm_mx_ptr("e2m1", a, a + 2, a, a, a * 64, 4, 16, 128) == 4     # SA alignment
    assert g.gemm_mx_ptr("e4m3", 0, a, a, a, a * 64, 4, 16, 128) == 1
    assert g.gemm_mx_ptr("e4m3", a, a, a, a, a + 64, 4, 16, 128) == 9         # C overlaps A
    assert g.gemm_mx_ptr("e4m3", a, a, a, a, a * 64, 0, 16, 128) == 0         # empty: nothing to do
