"""The C-ABI library loads, exports what include/tgemm.h declares, and its
host-side logic (argument checks, planning) behaves — no GPU needed."""

import json
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tgemm.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "page2_smem_exercises.json")


@pytest.fixture(scope="module")
def tg():
    from tiled_fp16_gemm_gb300 import build
    build.build()
    import tiled_fp16_gemm_gb300 as t
    t.library()
    return t


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(tg_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_expected_entry_points(tg):
    assert set(header_functions()) == set(tg.EXPORTS)


def test_library_exports_every_declared_symbol(tg):
    lib = tg.library()
    for name in header_functions():
        assert hasattr(lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", tg.LIB_PATH], capture_output=True,
                        text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r"\sT\s+(\S+)", nm.stdout))
        for name in header_functions():
            assert name in exported, name


def test_version_and_status_strings(tg):
    assert tg.tg_version().startswith("libtgemm ")
    assert "sm_103a" in tg.tg_version()
    for code in range(7):
        assert tg.tg_status_string(code).startswith("TG_")
    assert tg.tg_status_string(99) == "TG_ERR_UNKNOWN"


GOOD = 1 << 20  # a 16-byte aligned fake address (never dereferenced on these paths)


@pytest.mark.parametrize("args,want", [
    # (A, B, C, M, N, K, lda, ldb, ldc, epi)
    ((GOOD, GOOD, GOOD, 4, 4, 4, 8, 8, 8, 2), 1),          # bad epilogue
    ((GOOD, GOOD, GOOD, -1, 4, 4, 8, 8, 8, 0), 1),         # negative M
    ((GOOD, GOOD, GOOD, 4, 4, -4, 8, 8, 8, 0), 1),         # negative K
    ((GOOD, GOOD, GOOD, 1 << 31, 4, 4, 8, 8, 8, 0), 1),    # M too large
    ((0, GOOD, GOOD, 4, 4, 4, 8, 8, 8, 0), 1),             # null A
    ((GOOD, 0, GOOD, 4, 4, 4, 8, 8, 8, 0), 1),             # null B
    ((GOOD, GOOD, 0, 4, 4, 4, 8, 8, 8, 0), 1),             # null C
    ((GOOD, GOOD, GOOD, 4, 4, 9, 8, 16, 8, 0), 1),         # lda < K
    ((GOOD, GOOD, GOOD, 4, 12, 4, 8, 8, 16, 0), 1),        # ldb < N
    ((GOOD, GOOD, GOOD, 4, 12, 4, 8, 16, 8, 0), 1),        # ldc < N
    ((GOOD + 1, GOOD, GOOD, 4, 4, 4, 8, 8, 8, 0), 2),      # A not even element-aligned
    ((GOOD, GOOD + 3, GOOD, 4, 4, 4, 8, 8, 8, 0), 2),      # B not even element-aligned
    ((GOOD, GOOD, GOOD + 5, 4, 4, 4, 8, 8, 8, 0), 2),      # C not even element-aligned
    ((GOOD + 2, GOOD, GOOD, 4, 4, 4, 8, 8, 8, 0), None),   # A off 16 B: staged, accepted
    ((GOOD, GOOD, GOOD + 4, 4, 4, 4, 8, 8, 8, 0), None),   # C off 16 B: staged, accepted
    ((GOOD, GOOD, GOOD, 4, 4, 9, 7, 8, 8, 0), 1),          # odd lda < K still rejected
    ((GOOD, GOOD, GOOD, 4, 4, 4, 12, 9, 11, 0), None),     # odd leading dimensions accepted
    ((GOOD, GOOD, GOOD, 0, 4, 4, 8, 8, 8, 0), 0),          # M == 0: no-op
    ((0, 0, 0, 4, 0, 4, 8, 8, 8, 1), 0),                   # N == 0: no-op, nothing checked
    ((0, 0, GOOD, 4, 4, 0, 0, 0, 8, 0), None),             # K == 0: A/B/lda/ldb ignored
])
@pytest.mark.parametrize("entry", ["tg_gemm_f16", "tg_gemm_f16_host"])
def test_argument_checks_before_any_cuda_call(tg, entry, args, want):
    """The device entry point and the host-buffer one share these checks."""
    st = getattr(tg, entry)(*args, None)
    if want is None:
        # valid arguments: on a machine without an sm_103 device the call
        # reaches the device check and stops there
        if _has_gpu():
            pytest.skip("valid call would launch")
        assert st == tg.TG_ERR_UNSUPPORTED_DEVICE
    else:
        assert st == want, (args, tg.tg_status_string(st))


@pytest.mark.parametrize("in_dt,out_dt,bias,resid,ldr,K,want", [
    # (input type, output type, bias address, residual address, ldr, K, status)
    (3, 0, 0, 0, 0, 4, 1),                  # unknown input type
    (2, 2, 0, 0, 0, 4, 1),                  # fp32 is an output type only
    (0, 1, 0, 0, 0, 4, 1),                  # fp16 in, bf16 out: not offered
    (1, 0, 0, 0, 0, 4, 1),                  # bf16 in, fp16 out: not offered
    (0, 0, 0, GOOD, 3, 4, 1),               # ldr < N
    (0, 0, GOOD + 2, 0, 0, 4, 2),           # bias not 4-byte aligned
    (0, 0, 0, GOOD + 1, 8, 4, 2),           # residual not element-aligned
    (0, 0, GOOD + 4, GOOD + 2, 9, 4, None),  # scalar-path bias and residual: accepted
    (1, 2, GOOD, GOOD, 8, 4, None),         # bf16 in, fp32 out
    (0, 2, GOOD, GOOD, 8, 0, None),         # K == 0 with bias and residual
])
def test_gemm_ex_argument_checks(tg, in_dt, out_dt, bias, resid, ldr, K, want):
    epi = tg.tg_epilogue_ex_t(0, out_dt, bias or None, resid or None, ldr)
    st = tg.tg_gemm_ex(in_dt, GOOD, GOOD, GOOD, 4, 4, K, 8, 8, 8, epi, None)
    if want is None:
        if _has_gpu():
            pytest.skip("valid call would launch")
        assert st == tg.TG_ERR_UNSUPPORTED_DEVICE
    else:
        assert st == want, tg.tg_status_string(st)


def test_gemm_ex_fp32_output_alignment(tg):
    # an fp32 C must be aligned to its 4-byte element; a 2-byte offset is not
    epi = tg.tg_epilogue_ex_t(0, tg.TG_DTYPE_F32, None, None, 0)
    assert tg.tg_gemm_ex(0, GOOD, GOOD, GOOD + 2, 4, 4, 4, 8, 8, 8, epi, None) == \
        tg.TG_ERR_MISALIGNED
    # bad activation and a NULL epilogue (plain GEMM) take the usual checks
    epi = tg.tg_epilogue_ex_t(5, 0, None, None, 0)
    assert tg.tg_gemm_ex(0, GOOD, GOOD, GOOD, 4, 4, 4, 8, 8, 8, epi, None) == \
        tg.TG_ERR_INVALID_VALUE
    assert tg.tg_gemm_ex(0, GOOD, GOOD, 0, 4, 4, 4, 8, 8, 8, None, None) == \
        tg.TG_ERR_INVALID_VALUE


@pytest.mark.parametrize("A,Bq,S,N,K,lda,ldbq,ldbs,want", [
    # M = 4 throughout; C = GOOD with ldc = N; K = 64 needs ldbq >= 32
    (GOOD, GOOD, GOOD, 32, 64, 64, 32, 32, None),        # valid
    (GOOD + 2, GOOD, GOOD, 32, 64, 67, 32, 32, None),    # A off 16 bytes, odd lda: staged
    (GOOD, GOOD + 8, GOOD, 32, 64, 64, 32, 32, 2),       # Bq not 16-byte aligned
    (GOOD, GOOD, GOOD + 4, 32, 64, 64, 32, 32, 2),       # scales not 16-byte aligned
    (GOOD, GOOD, GOOD, 32, 64, 64, 40, 32, 2),           # ldbq not a multiple of 16
    (GOOD, GOOD, GOOD, 32, 64, 64, 32, 40, 2),           # ldbs not a multiple of 16
    (GOOD, GOOD, GOOD, 32, 80, 80, 32, 32, 1),           # ldbq < ceil(K/2) = 40
    (GOOD, GOOD, GOOD, 40, 64, 64, 32, 32, 1),           # ldbs < N
    (GOOD, 0, GOOD, 32, 64, 64, 32, 32, 1),              # null Bq
    (GOOD, GOOD, 0, 32, 64, 64, 32, 32, 1),              # null scales
    (GOOD + 1, GOOD, GOOD, 32, 64, 64, 32, 32, 2),       # A not element-aligned
    (0, 0, 0, 32, 0, 0, 0, 0, None),                     # K == 0: operands ignored
])
def test_gemm_mxfp4_argument_checks(tg, A, Bq, S, N, K, lda, ldbq, ldbs, want):
    st = tg.tg_gemm_mxfp4(A, Bq, S, GOOD, 4, N, K, lda, ldbq, ldbs, N, None, None)
    if want is None:
        if _has_gpu():
            pytest.skip("valid call would launch")
        assert st == tg.TG_ERR_UNSUPPORTED_DEVICE
    else:
        assert st == want, tg.tg_status_string(st)


def test_gemm_mxfp4_epilogue_checks(tg):
    bf16_out = tg.tg_epilogue_ex_t(0, tg.TG_DTYPE_BF16, None, None, 0)  # input is fp16
    assert tg.tg_gemm_mxfp4(GOOD, GOOD, GOOD, GOOD, 4, 32, 64, 64, 32, 32, 32, bf16_out,
                            None) == tg.TG_ERR_INVALID_VALUE
    bad_act = tg.tg_epilogue_ex_t(3, tg.TG_DTYPE_F16, None, None, 0)
    assert tg.tg_gemm_mxfp4(GOOD, GOOD, GOOD, GOOD, 4, 32, 64, 64, 32, 32, 32, bad_act,
                            None) == tg.TG_ERR_INVALID_VALUE
    short_r = tg.tg_epilogue_ex_t(0, tg.TG_DTYPE_F16, None, GOOD, 16)  # ldr < N
    assert tg.tg_gemm_mxfp4(GOOD, GOOD, GOOD, GOOD, 4, 32, 64, 64, 32, 32, 32, short_r,
                            None) == tg.TG_ERR_INVALID_VALUE


@pytest.mark.parametrize("args,want", [
    # (in_dtype, Ac, E, B, C, M, N, K, ldac, lde, ldb, ldc)
    ((0, GOOD, GOOD, GOOD, GOOD, 4, 16, 64, 32, 4, 16, 16), None),    # valid
    ((0, GOOD, GOOD, GOOD, GOOD, 4, 16, 48, 24, 4, 16, 16), 1),       # K not a multiple of 32
    ((0, GOOD, GOOD, GOOD, GOOD, 4, 16, 64, 24, 4, 16, 16), 1),       # ldac < K/2
    ((0, GOOD, GOOD, GOOD, GOOD, 4, 16, 64, 32, 1, 16, 16), 1),       # lde < K/32
    ((0, GOOD, GOOD, GOOD, GOOD, 4, 16, 64, 40, 6, 16, 16), 2),       # lde not a multiple of 4
    ((0, GOOD, GOOD, GOOD, GOOD, 4, 16, 64, 36, 4, 16, 16), 2),       # ldac not a multiple of 8
    ((0, GOOD + 8, GOOD, GOOD, GOOD, 4, 16, 64, 32, 4, 16, 16), 2),   # Ac not 16-byte aligned
    ((0, GOOD, GOOD, GOOD, GOOD + 2, 4, 16, 64, 32, 4, 16, 16), 2),   # C not 16-byte aligned
    ((0, GOOD, 0, GOOD, GOOD, 4, 16, 64, 32, 4, 16, 16), 1),          # null metadata
    ((3, GOOD, GOOD, GOOD, GOOD, 4, 16, 64, 32, 4, 16, 16), 1),       # unknown type
    ((1, 0, 0, 0, GOOD, 4, 16, 0, 0, 0, 0, 16), None),                # K == 0, bf16
])
def test_gemm_sp24_argument_checks(tg, args, want):
    st = tg.tg_gemm_sp24(*args, None, None)
    if want is None:
        if _has_gpu():
            pytest.skip("valid call would launch")
        assert st == tg.TG_ERR_UNSUPPORTED_DEVICE
    else:
        assert st == want, tg.tg_status_string(st)


def test_noalloc_keeps_the_tma_layout_rule(tg):
    # the entry point without allocation has no staging buffer
    st = tg.tg_gemm_f16_noalloc(GOOD, GOOD, GOOD, 4, 4, 4, 12, 8, 8, 0, None)
    assert st == tg.TG_ERR_MISALIGNED
    st = tg.tg_gemm_f16_noalloc(GOOD + 2, GOOD, GOOD, 4, 4, 4, 8, 8, 8, 0, None)
    assert st == tg.TG_ERR_MISALIGNED


def test_valid_call_without_gpu_reports_unsupported_device(tg):
    if _has_gpu():
        pytest.skip("a GPU is present")
    assert tg.tg_gemm_f16(GOOD, GOOD, GOOD, 4, 4, 4, 8, 8, 8, 0, None) == tg.TG_ERR_UNSUPPORTED_DEVICE
    assert tg.tg_sync_status(None) == tg.TG_ERR_UNSUPPORTED_DEVICE


def test_ring_bytes_reproduces_page_exercises(tg):
    g = json.load(open(GOLDEN))
    for c in g["cases"]:
        assert tg.tg_ring_bytes(c["block_M"], c["block_N"], c["block_K"], c["stages"],
                                c["elem_bytes"]) == c["ring_bytes"]
    # one A stage, and the B buffers following three A stages
    assert tg.tg_ring_bytes(128, 128, 64, 1, 2) == 2 * g["a_stage_bytes"]
    assert 3 * g["a_stage_bytes"] == g["b_buffer_offset_3_stages"]
    assert (228 * 1024) // tg.tg_ring_bytes(128, 128, 64, 3, 2) == g["blocks_per_sm_in_228KB_3_stages"]
    assert tg.tg_ring_bytes(0, 128, 64, 3, 2) == -1


def test_plan_k_steps_and_grid_match_page_listing(tg):
    g = json.load(open(GOLDEN))
    p = tg.tg_plan_f16(1024, 1024, 1024, 152)
    assert p.k_blocks == g["k_steps_for_K1024_BK64"]
    assert p.bk == 64
    # with 128×128 tiles the page's grid is (N/128, M/128)
    assert (1024 // 128, 1024 // p.bm) == tuple(g["grid_for_M_N_1024_tile_128"])


def test_plans(tg):
    p = tg.tg_plan_f16(8192, 28672, 4096, 152)
    assert p.kernel == tg.TG_KERNEL_PERSISTENT and p.cluster == 2
    assert (p.bm, p.bn, p.bk, p.mma_m, p.mma_n) == (256, 256, 128, 256, 256)
    assert p.num_tiles == 32 * 112 and p.grid == 152 and p.k_blocks == 32 and p.stages == 3
    assert p.smem_bytes <= 232448  # 227 KB opt-in limit per CTA
    assert p.ring_bytes == 2 * tg.tg_ring_bytes(128, 128, 128, p.stages, 2)
    one = tg.tg_plan_f16(1536, 1536, 4096, 152)  # 144 tiles of 128x128 fit one wave
    assert one.cluster == 1 and (one.bm, one.bn) == (128, 128) and one.grid == 144
    # 64 pair tiles (< 76 pairs) but 256 tiles of 128x128 (> 152 SMs), K >= 1024: pairs
    sub = tg.tg_plan_f16(2048, 2048, 4096, 152)
    assert sub.cluster == 2 and sub.num_tiles == 64 and sub.grid == 128
    short = tg.tg_plan_f16(2048, 2048, 512, 152)  # short K: one-CTA 128x128 tiles
    assert short.cluster == 1 and (short.bm, short.bn) == (128, 128)
    pair = tg.tg_plan_f16(2048, 4864, 4096, 152)  # 8 x 19 = 152 pair tiles: two waves of pairs
    assert pair.cluster == 2 and pair.num_tiles == 152 and pair.grid == 152
    s = tg.tg_plan_f16(64, 16384, 8192, 152)
    assert s.kernel == tg.TG_KERNEL_SKINNY
    assert (s.mma_m, s.mma_n) == (128, 64) and s.tiles_n == 128
    assert (s.bk, s.k_blocks, s.stages) == (64, 128, 9)
    # 128 tiles: one CTA per whole tile (no partial sums)
    assert s.grid == 128 and s.split_k == 1 and s.workspace_bytes > 0
    assert s.smem_bytes <= 232448
    # 224 tiles: two whole tiles per CTA; 64 tiles: two equal k pieces each;
    # 86 tiles (no aligned grid reaches 0.7 of the SMs): balanced over 152
    assert tg.tg_plan_f16(128, 28672, 4096, 152).grid == 112
    h = tg.tg_plan_f16(64, 8192, 8192, 152)
    assert h.grid == 128 and h.split_k == 2
    assert tg.tg_plan_f16(64, 11008, 4096, 152).grid == 152
    w = tg.tg_plan_f16(128, 16384, 8192, 152)  # Mp = 128: 64-k units, 6 stages
    assert w.kernel == tg.TG_KERNEL_SKINNY and (w.bk, w.k_blocks, w.stages) == (64, 128, 6)
    assert w.smem_bytes <= 232448
    small = tg.tg_plan_f16(7, 5, 3, 152)
    assert small.kernel == tg.TG_KERNEL_SKINNY and small.mma_n == 16 and small.grid == 1
    assert tg.tg_plan_f16(0, 5, 3, 152).kernel == tg.TG_KERNEL_NONE
    assert tg.tg_plan_f16(5, 5, 0, 152).kernel == tg.TG_KERNEL_FILL
    mid = tg.tg_plan_f16(1024, 1024, 1024, 152)  # 64 tiles of 128x128 would fill < half
    assert mid.kernel == tg.TG_KERNEL_PERSISTENT and mid.bn == 64 and mid.num_tiles == 128
    wide = tg.tg_plan_f16(1536, 1024, 1024, 152)  # 96 tiles of 128x128: more than half
    assert wide.kernel == tg.TG_KERNEL_PERSISTENT and wide.bn == 128 and wide.num_tiles == 96
    with pytest.raises(tg.TgemmError):
        tg.tg_plan_f16(-1, 5, 5, 152)
    with pytest.raises(tg.TgemmError):
        tg.tg_plan_f16(5, 5, 5, 0)


def test_tile_order_is_a_bijection_and_grouped(tg):
    p = tg.tg_plan_f16(8192, 28672, 4096, 152)
    seen = set()
    for t in range(p.num_tiles):
        seen.add(tg.tg_tile_coord(p, t))
    assert len(seen) == p.num_tiles
    assert all(0 <= m < p.tiles_m and 0 <= n < p.tiles_n for m, n in seen)
    # the first wave (one tile per CTA pair) spans group_m row blocks and few column blocks
    wave = p.grid // p.cluster
    first = [tg.tg_tile_coord(p, t) for t in range(wave)]
    assert len({m for m, _ in first}) == p.group_m
    assert len({n for _, n in first}) <= -(-wave // p.group_m)
    with pytest.raises(tg.TgemmError):
        tg.tg_tile_coord(p, p.num_tiles)


def test_schedule_bruteforce_cpp(tmp_path):
    exe = os.path.join(str(tmp_path), "sched_check")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I",
                    os.path.join(ROOT, "tiled_fp16_gemm_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "sched_check.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout


def test_skinny_grid_invariants(tg):
    """The M <= 128 planner over a sweep of shapes: at most one CTA per SM,
    at least 8 units of work per CTA (unless the problem is smaller), an
    aligned grid cuts only at tile edges or equal tile fractions, and the
    cluster launch is asked for exactly when each tile has four k-pieces."""
    for M in (1, 16, 64, 100, 128):
        for N in (1, 128, 1000, 2048, 4096, 4864, 5120, 8192, 11008, 14336, 16384, 28672):
            for K in (64, 1000, 4096, 8192, 14336):
                p = tg.tg_plan_f16(M, N, K, 152)
                assert p.kernel == tg.TG_KERNEL_SKINNY
                T, KB, G = p.tiles_n, p.k_blocks, p.grid
                U = T * KB
                assert 1 <= G <= 152
                assert G * 8 <= U or G == 1, (M, N, K, G, U)
                assert p.cluster in (1, 4)
                if p.cluster == 4:
                    assert G == 4 * T and KB // 4 >= 8, (M, N, K)
                if G < T and T % G == 0 and G * 10 >= 152 * 7:
                    assert p.split_k == 1  # whole tiles per CTA
                if G == T * (G // T) and G > T and G * 10 >= 152 * 7 and p.cluster == 4:
                    assert p.split_k == 4


def test_pair_split_invariants(tg):
    """The pair planner over a sweep of shapes: an even grid of at most 152
    CTAs, and a last wave cut either into two column halves per tile or into
    at most 4 k-pieces per tile, each at least 8 blocks of 128 k, that fit
    the idle pairs."""
    for M in (256, 1000, 2048, 2560, 4096, 8192):
        for N in (256, 1000, 2048, 4096, 4864, 8192, 11008, 28672):
            for K in (512, 1024, 4096, 8192, 16384):
                p = tg.tg_plan_f16(M, N, K, 152)
                if p.cluster != 2:
                    continue
                T, KB, G = p.num_tiles, p.k_blocks, p.grid
                P = G // 2
                assert G % 2 == 0 and 2 <= G <= 152
                S, H = p.split_k, p.split_n
                assert 1 <= S <= 4 and H in (1, 2) and (S == 1 or H == 1)
                R = T % P if T >= P else T
                if S > 1:
                    assert KB // S >= 8 and R * S <= P, (M, N, K, S)
                    assert p.workspace_bytes > 0
                elif H > 1:
                    assert 2 * R <= P and p.workspace_bytes == 0, (M, N, K)
                else:
                    assert P == min(T, 76)
                    assert R == 0 or 2 * R > P, (M, N, K)  # halves would have fit


def test_plan_limits(tg):
    """tg_plan_f16_limits: with the nominal limits it is tg_plan_f16; with
    fewer resident pairs or four-CTA clusters it plans only what fits."""
    for shape in [(8192, 28672, 4096), (4096, 4096, 4096), (2048, 2048, 4096),
                  (1024, 1024, 1024), (64, 4096, 4096), (64, 16384, 8192), (7, 5, 3),
                  (5, 5, 0)]:
        a = tg.tg_plan_f16(*shape, 152)
        b = tg.tg_plan_f16_limits(*shape, 152, 76, 38, 38)
        assert bytes(a) == bytes(b), shape
    # fewer pairs fit at once: the grid stays within them, the tail split follows
    p = tg.tg_plan_f16_limits(8192, 28672, 4096, 152, 74, 38, 38)
    assert p.cluster == 2 and p.grid <= 148 and p.grid % 2 == 0
    R = p.num_tiles % (p.grid // 2)
    assert R * p.split_k * p.split_n <= p.grid // 2
    # limits above num_sms / 2 are clamped to it
    assert bytes(tg.tg_plan_f16_limits(8192, 28672, 4096, 152, 99, 38, 38)) == \
        bytes(tg.tg_plan_f16(8192, 28672, 4096, 152))
    # no pair fits: one-CTA tiles
    p = tg.tg_plan_f16_limits(8192, 28672, 4096, 152, 0, 38, 38)
    assert p.kernel == tg.TG_KERNEL_PERSISTENT and p.cluster == 1
    # a skinny grid of four-piece clusters: launched without clusters unless
    # every cluster fits at once
    s = tg.tg_plan_f16(64, 4096, 4096, 152)
    assert s.cluster == 4 and s.grid == 128
    s2 = tg.tg_plan_f16_limits(64, 4096, 4096, 152, 76, 31, 38)
    assert s2.cluster == 1 and s2.grid == 128 and s2.split_k == s.split_k
    assert tg.tg_plan_f16_limits(64, 4096, 4096, 152, 76, 32, 0).cluster == 4
    w = tg.tg_plan_f16(128, 4096, 14336, 152)
    assert w.cluster == 4
    assert tg.tg_plan_f16_limits(128, 4096, 14336, 152, 76, 38, 31).cluster == 1
    with pytest.raises(tg.TgemmError):
        tg.tg_plan_f16_limits(5, 5, 5, 152, -1, 38, 38)
