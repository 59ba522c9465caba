"""Host-side checks (no GPU): the library loads and exports the declared ABI, and the
planner / raster / stream-K / traffic-model logic matches the pages' numbers."""
import os
import re

import numpy as np
import pytest

import dense_gemm_sm_gb300 as dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dgemm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M)) - {"if"})


def test_library_exports_every_declared_symbol():
    lib = dg.load()
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/dgemm.h but not exported"
    assert set(names) == set(dg.EXPORTED)


def test_status_strings():
    for s in range(7):
        assert dg.status_string(s).startswith("DG_")


def test_plan_dispatch_table():
    ffn = dg.dg_plan_gemm(1, 1024, 12288, 4096, num_sms=152)
    # FFN on CTA pairs: 256 x 256 tiles, 4 x 48 of them, 76 pairs of CTAs.
    assert ffn["kernel"] == dg.DG_KERNEL_TC2_BF16 and ffn["tile_m"] == 256 and ffn["tile_n"] == 256
    assert ffn["tiles"] == 192 and ffn["grid"] == 152
    for m in (1, 4, 16):
        p = dg.dg_plan_gemm(1, m, 12288, 4096, num_sms=152)
        assert p["kernel"] == dg.DG_KERNEL_THIN_BF16 and p["ntok"] == 16
    assert dg.dg_plan_gemm(1, 32, 12288, 4096, num_sms=152)["ntok"] == 32
    assert dg.dg_plan_gemm(1, 33, 12288, 4096, num_sms=152)["kernel"] == dg.DG_KERNEL_TC_BF16
    qk = dg.dg_plan_gemm(1, 2048, 2048, 128, batch=64, op_b=dg.DG_OP_T, c_type=dg.DG_OUT_F32,
                         num_sms=152)
    assert qk["kernel"] == dg.DG_KERNEL_TC_BF16 and qk["tiles"] == 64 * 16 * 8
    assert dg.dg_plan_gemm(0, 4096, 4096, 4096, num_sms=152)["kernel"] == dg.DG_KERNEL_SIMT_F32
    # Stream-K tail of the tile kernel: on for FFN (2 whole waves of K = 4096 + 40 tail
    # pair tiles, spread over all 76 pairs; partials and counters per CTA of a pair); off
    # where the whole waves are too short to hide the combine (one wave of K = 1024) or a
    # tile has too few K blocks (QK^T, K = 128).
    assert ffn["tail_tiles"] == 40 and ffn["splits"] == 76
    assert ffn["workspace_bytes"] == 2 * 76 * 2 * 128 * 256 * 4 + 2 * 40 * 4
    sk = dg.dg_plan_gemm(1, 1280, 4096, 6144, num_sms=152)
    assert sk["tail_tiles"] == 4 and sk["splits"] == 16            # 4 pairs per tail tile
    assert dg.dg_plan_gemm(1, 1280, 4096, 1024, num_sms=152)["tail_tiles"] == 0
    assert qk["tail_tiles"] == 0
    assert dg.dg_plan_gemm(1, 2048, 2048, 4096, num_sms=152)["tail_tiles"] == 0  # one partial wave
    # Single CTAs where a pair would waste its second CTA (one 128-row tile row) or a batch.
    assert dg.dg_plan_gemm(1, 128, 8192, 4096, num_sms=152)["kernel"] == dg.DG_KERNEL_TC_BF16
    assert dg.dg_plan_gemm(1, 129, 8192, 4096, num_sms=152)["kernel"] == dg.DG_KERNEL_TC2_BF16
    assert dg.dg_plan_gemm(0, 10, 10, 0, num_sms=152)["kernel"] == dg.DG_KERNEL_SCALE
    assert dg.dg_plan_gemm(1, 0, 10, 10, num_sms=152)["kernel"] == dg.DG_KERNEL_NONE


def test_plan_fp8_pair_width():
    # FP8 pairs take the width (256 or 224) with the smaller tile-waves x width, 256 on a tie.
    # FFN shape: 4 x 48 tiles of 256 = 3 waves of 76 pairs (768) vs 4 x 55 of 224 (672).
    ffn = dg.dg_plan_gemm(2, 1024, 12288, 4096, num_sms=152)
    assert ffn["kernel"] == dg.DG_KERNEL_TC2_BF16 and ffn["tile_n"] == 224 and ffn["tiles"] == 220
    # FP8 pairs stage one 128-byte K atom (BF16 pairs two).
    assert ffn["tile_k"] == 128 and ffn["kblocks"] == 32 and ffn["tail_tiles"] == 0 and ffn["stages"] == 6
    # Example 5-8 GEMM: 16 x 6 tiles (2 waves, 512) vs 16 x 7 (2 waves, 448).
    assert dg.dg_plan_gemm(2, 4096, 1536, 4096, num_sms=152)["tile_n"] == 224
    # 2 x 35 tiles of 256 fit one wave; 2 x 40 of 224 would need two.
    assert dg.dg_plan_gemm(2, 512, 8960, 4096, num_sms=152)["tile_n"] == 256
    # K = 6144 gives the 224-wide tiles a stream-K tail: 220 = 2 x 76 + 68.
    sk = dg.dg_plan_gemm(2, 1024, 12288, 6144, num_sms=152)
    assert sk["tile_n"] == 224 and sk["tail_tiles"] == 68 and sk["splits"] == 76
    assert sk["workspace_bytes"] == 2 * 76 * 2 * 128 * 224 * 4 + 2 * 68 * 4
    # The BF16 path keeps 256 on pairs; one 128-row tile row keeps single CTAs.
    assert dg.dg_plan_gemm(1, 1024, 12288, 4096, num_sms=152)["tile_n"] == 256
    assert dg.dg_plan_gemm(2, 128, 12288, 4096, num_sms=152)["kernel"] == dg.DG_KERNEL_TC_BF16
    with pytest.raises(RuntimeError):
        dg.dg_plan_gemm(2, 1024, 1024, 1024, batch=2, num_sms=152)


def test_tile_width_choice():
    # 256-wide tiles except for narrow problems (measured sweep; see the planner's comment)
    for M, N, batch in [(1024, 12288, 1), (4096, 4096, 1), (2048, 2048, 64), (300, 1000, 1),
                        (8192, 8192, 1), (64, 136, 1)]:
        assert dg.dg_plan_gemm(1, M, N, 512, batch=batch, num_sms=152)["tile_n"] == 256
    assert dg.dg_plan_gemm(1, 4096, 128, 512, num_sms=152)["tile_n"] == 128
    assert dg.dg_plan_gemm(1, 4096, 96, 512, num_sms=152)["tile_n"] == 128


@pytest.mark.parametrize("tiles_m,tiles_n,group", [(10, 10, 8), (8, 48, 8), (32, 16, 8), (3, 7, 8),
                                                    (17, 5, 4), (1, 1, 8), (9, 1, 8)])
def test_raster_is_a_bijection(tiles_m, tiles_n, group):
    # Swizzle bijection and range property (MUSA lesson m11-l5, Block ID Swizzle discussion).
    batch = 2
    seen = set()
    for t in range(batch * tiles_m * tiles_n):
        b, tm, tn = dg.dg_raster_tile(t, tiles_m, tiles_n, group)
        assert 0 <= b < batch and 0 <= tm < tiles_m and 0 <= tn < tiles_n
        seen.add((b, tm, tn))
    assert len(seen) == batch * tiles_m * tiles_n


def test_raster_locality_matches_swizzle_example():
    # MUSA lesson m11-l5: changing row every 8 blocks, 64 blocks need 8 tile_m and 8 tile_n
    # operand tiles: amplification (64+64)/(8+8) = 8 versus ~2 for the plain row order.
    tiles_m, tiles_n = 64, 64
    for start in range(0, tiles_m * tiles_n, 64):
        ids = [dg.dg_raster_tile(t, tiles_m, tiles_n, 8) for t in range(start, start + 64)]
        rows = {tm for _, tm, _ in ids}
        cols = {tn for _, _, tn in ids}
        assert len(rows) == 8 and len(cols) == 8
        assert (64 + 64) / (len(rows) + len(cols)) == 8


def test_streamk_partition_covers_units_once():
    for units, ctas in [(6144, 152), (96, 152), (7, 3), (1000, 152), (152, 152)]:
        starts = [dg.dg_streamk_start(c, units, ctas) for c in range(ctas + 1)]
        assert starts[0] == 0 and starts[-1] == units
        assert all(a <= b for a, b in zip(starts, starts[1:]))
        sizes = [b - a for a, b in zip(starts, starts[1:])]
        assert max(sizes) - min(sizes) <= 1


def read_tile_table():
    rows = []
    for line in open(os.path.join(GOLDEN, "tile_traffic.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append([float(x) for x in line.split()])
    return rows


def test_tile_traffic_model_reproduces_pages_table():
    # "Operator & Runtime" section 5.2.2, Example 5-3 and its table (k = 32).
    M, K, N = 1024, 4096, 12288
    flops = 2 * M * N * K
    for m, n, kib, mib, intensity in read_tile_table():
        assert dg.dg_model_local_bytes(int(m), int(n), 32, 2) == kib * 1024
        v = dg.dg_model_traffic_bytes(M, N, K, int(m), int(n), 2, 2)
        assert v == mib * 2 ** 20
        assert abs(flops / v - intensity) < 0.06


def test_ffn_counts_from_chapter_intro():
    # 128 MiB once-through bytes = the traffic model with one tile covering everything.
    v = dg.dg_model_traffic_bytes(1024, 12288, 4096, 1024, 12288, 2, 2)
    assert v == 128 * 2 ** 20


def test_quant_traffic_model_reproduces_example_5_8():
    from .test_oracle_pins import read_golden
    # "Operator & Runtime" section 5.4.4, Example 5-8: A FP16 [4096, 4096], FP8 weights
    # [4096, 1536], FP16 output, 128 x 128 tiles: 444 MiB with separate quantisation, 620 MiB
    # fused into the GEMM (tests/golden/fp8_e4m3.txt).
    g, _ = read_golden("fp8_e4m3.txt")
    MiB = 2.0 ** 20
    sep = dg.dg_model_quant_traffic_bytes(4096, 4096, 1536, 128, 128, 2, 1, 2, fused=False)
    fus = dg.dg_model_quant_traffic_bytes(4096, 4096, 1536, 128, 128, 2, 1, 2, fused=True)
    assert sep / MiB == g["total_separate_mib"] and fus / MiB == g["total_fused_mib"]
    wo = dg.dg_model_quant_traffic_bytes(4096, 0, 1536, 128, 128, 2, 1, 2) / MiB     # output only
    assert wo == 12
    # weights + output = 204 MiB in both; the input side 240 vs 416 MiB
    w_out = 32 * 6 + 12
    assert w_out == g["weights_output_mib"]
    assert sep / MiB - w_out == g["input_separate_mib"] and fus / MiB - w_out == g["input_fused_mib"]


def test_fp32_plan_small_and_streamk():
    # 256^3: 4 tiles of 128 x 128 for 2 x 152 resident CTAs -- the small-tile kernel, 64
    # tiles of 32 x 32, K = 256 in one chunk (two staged pieces of 128).
    p = dg.dg_plan_gemm(0, 256, 256, 256, num_sms=152)
    assert (p["tile_m"], p["tiles"], p["splits"], p["grid"], p["kblocks"]) == (32, 64, 1, 64, 2)
    assert p["workspace_bytes"] == 0
    # 200 x 136 x 1000: 35 small tiles, K cut in 2 chunks of at least 4 pieces.
    p = dg.dg_plan_gemm(0, 200, 136, 1000, num_sms=152)
    assert (p["tile_m"], p["tiles"], p["splits"], p["grid"]) == (32, 35, 2, 70)
    assert p["workspace_bytes"] == 35 * 2 * 32 * 32 * 4 + 35 * 4
    assert dg.dg_plan_gemm(0, 7, 9, 5, num_sms=152)["splits"] == 1      # one K piece: no split
    # 1000 x 3000 x 777: 192 tiles x 25 K tiles for 304 resident CTAs -- stream-K, 15.8 K
    # tiles per CTA (splits 0); 4096^3 keeps whole-tile waves and a split tail.
    p = dg.dg_plan_gemm(0, 1000, 3000, 777, num_sms=152)
    assert (p["tiles"], p["splits"], p["grid"], p["tail_tiles"]) == (192, 0, 304, 192)
    p = dg.dg_plan_gemm(0, 4096, 4096, 4096, num_sms=152)
    assert (p["tiles"], p["splits"], p["tail_tiles"]) == (1024, 8, 112)


def _cdiv(a, b):
    return -(-a // b)


def test_plan_properties_on_random_shapes():
    # Invariants of the planner over seeded random shapes, recomputed here from the tile
    # sizes: tile counts, grids, the FP32 small-tile, tail-split and stream-K schedules, the
    # decode stream-K grid, CTA pairs and their widths, stream-K tails and workspace sizes.
    rng = np.random.default_rng(20261202)
    sms = 152
    for _ in range(1500):
        M = int(rng.choice([rng.integers(1, 40), rng.integers(1, 5000), rng.integers(1, 70000)]))
        N = int(rng.choice([rng.integers(1, 300), rng.integers(1, 20000)]))
        K = int(rng.choice([rng.integers(1, 200), rng.integers(1, 9000)]))
        batch = int(rng.choice([1, 1, 1, rng.integers(2, 70)]))
        _check_f32_plan(M, N, K, batch, sms)
        _check_bf16_fp8_plans(M, N, K, batch, sms)


def _check_f32_plan(M, N, K, batch, sms):
    p = dg.dg_plan_gemm(0, M, N, K, batch=batch, num_sms=sms)
    assert p["kernel"] == dg.DG_KERNEL_SIMT_F32
    tiles = batch * _cdiv(M, 128) * _cdiv(N, 128)
    G = 2 * sms
    if 4 * tiles <= G:
        # Small-tile kernel: 32 x 32 tiles, K in 128-wide pieces, chunks of at least 4
        # pieces, at most 16 chunks, at most as many chunk CTAs as are resident.
        t32 = batch * _cdiv(M, 32) * _cdiv(N, 32)
        pieces = _cdiv(K, 128)
        S = max(1, min(G // t32, _cdiv(pieces, 4), 16))
        assert (p["tile_m"], p["tile_n"], p["tile_k"]) == (32, 32, 128)
        assert (p["tiles"], p["kblocks"], p["splits"], p["grid"]) == (t32, pieces, S, t32 * S)
        assert p["workspace_bytes"] == (t32 * S * 4096 + t32 * 4 if S > 1 else 0)
        return
    KT = _cdiv(K, p["tile_k"])
    assert p["tiles"] == tiles and p["kblocks"] == KT
    if tiles < G and tiles * KT >= 4 * G and _cdiv(tiles * KT, G) <= 7 * KT:
        # Stream-K: tiles for between a quarter and one wave, at least 4 K tiles per
        # resident CTA, ranges of at most 7 tiles' K (so at most 8 segments); one wave of
        # CTAs over all tiles.
        assert p["splits"] == 0 and p["grid"] == G and p["tail_tiles"] == tiles
        assert p["workspace_bytes"] == 2 * G * 16 * 256 * 16 + tiles * 4
        return
    assert p["splits"] >= 1 and 0 <= p["tail_tiles"] <= tiles
    assert p["grid"] == tiles - p["tail_tiles"] + p["tail_tiles"] * p["splits"]
    if p["splits"] > 1:
        # Chunks of at least 256 of K (8 K tiles), at most 3 waves of chunk CTAs on the
        # 2 x 152 resident slots.
        assert p["tail_tiles"] > 0 and p["tail_tiles"] * p["splits"] <= 3 * G
        assert p["splits"] <= p["kblocks"] // 8
        assert p["workspace_bytes"] > 0
    else:
        assert p["tail_tiles"] == 0 and p["workspace_bytes"] == 0


def _check_bf16_fp8_plans(M, N, K, batch, sms):
    # BF16 and FP8 (FP8 is planned for one problem only)
    for dtype in (1, 2) if batch == 1 else (1,):
        q = dg.dg_plan_gemm(dtype, M, N, K, batch=batch, num_sms=sms)
        if dtype == 1 and batch == 1 and M <= 32:
            assert q["kernel"] == dg.DG_KERNEL_THIN_BF16
            assert q["ntok"] == (16 if M <= 16 else 32)
            units = _cdiv(N, 128) * _cdiv(K, 64)
            assert q["tiles"] == _cdiv(N, 128) and q["grid"] == min(units, sms)
            continue
        pair = q["kernel"] == dg.DG_KERNEL_TC2_BF16
        ka = 2 if pair and dtype == 1 else 1  # 128-byte K atoms per stage
        tk = (128 if dtype == 2 else 64) * ka
        assert q["tile_k"] == tk and q["kblocks"] == _cdiv(K, tk)
        assert q["stages"] == ((3 if ka == 2 else 6) if pair else (4 if q["tile_n"] >= 192 else 6))
        bn = q["tile_n"]
        if q["kernel"] == dg.DG_KERNEL_TC2_BF16:
            assert batch == 1 and _cdiv(M, 128) >= 2 and q["tile_m"] == 256
            tm2 = _cdiv(_cdiv(M, 128), 2)
            assert q["tiles"] == tm2 * _cdiv(N, bn)
            assert q["grid"] % 2 == 0 and q["grid"] // 2 == min(q["tiles"], sms // 2)
            if dtype == 2:
                w256 = _cdiv(tm2 * _cdiv(N, 256), sms // 2) * 256
                w224 = _cdiv(tm2 * _cdiv(N, 224), sms // 2) * 224
                assert bn == (224 if w224 < w256 else 256)
            else:
                assert bn == 256
            G = q["grid"] // 2
        else:
            assert q["kernel"] == dg.DG_KERNEL_TC_BF16 and q["tile_m"] == 128
            assert q["tiles"] == batch * _cdiv(M, 128) * _cdiv(N, bn)
            assert q["grid"] == min(q["tiles"], sms)
            G = q["grid"]
        if q["tail_tiles"]:
            # thresholds in 128-byte K atoms
            assert q["tiles"] > G and q["tail_tiles"] == q["tiles"] % G
            assert q["kblocks"] * ka >= 16 and (q["tiles"] // G) * q["kblocks"] * ka >= 96
            assert 1 <= q["splits"] <= min(4 * q["tail_tiles"], G)
            assert q["workspace_bytes"] > 0
        else:
            assert q["splits"] == 1


