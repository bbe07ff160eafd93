"""The bench line's fixed arithmetic: rows per step, algorithmic bytes and flops per call (the
roofline numerators), launches per step and the profiled traffic, worked out by hand for the
8B-shaped token step and the 1M-workspace block step."""
import bench
import synth

TW, BW = synth.TOKEN[bench.TOKEN_WL], synth.BLOCK[bench.BLOCK_WL]


def test_workloads_are_the_documented_ones():
    assert (TW.L, TW.Hq, TW.Hkv, TW.D, TW.N) == (36, 32, 8, 128, 32768)
    assert (BW.L, BW.Hq, BW.Hkv, BW.D, BW.n_blocks, BW.M) == (64, 40, 8, 128, 32768, 2048)


def test_rows_per_step():
    # token: L * Hkv * |H| = 36 * 8 * 32000; block: L * Hkv * |C| = 64 * 8 * 32636
    assert bench.workload_rows(TW, BW) == (9_216_000, 16_709_632)


def test_algorithmic_amounts():
    a = bench.kernel_algorithmic(TW, BW)
    # candidate K rows once (36 * 32000 * 8 * 256 B) plus the rule vector
    assert a["rule_scores"] == ("hbm", 2_359_296_000 + 32768 * 4)
    # the turn's query rows (36 * 32 * 256 * 256 B) plus M read and written
    assert a["memory_update"] == ("hbm", 75_497_472 + 2 * 36 * 32 * 128 * 4)
    # 4096 new raw tokens of every (layer, kv head) read, 128 index rows written
    assert a["meank_build"] == ("hbm", 64 * 8 * 4096 * 256 + 64 * 8 * 128 * 256)
    # 2048 blocks x 32 tokens of every (layer, kv head), read and written
    assert a["rerope_scatter"] == ("hbm", 2 * 64 * 8 * 2048 * 32 * 256)
    # one QK^T over the candidates: 2 * L * Hq * M * |C| * D
    assert a["block_scores"] == ("tensor", 43_803_297_710_080)


def test_launches_and_traffic():
    assert sum(bench.LAUNCHES.values()) == 13
    assert bench.LAUNCHES["block_scores"] == 4 and bench.LAUNCHES["rule_scores"] == 3
    assert abs(bench.PROFILED_TRAFFIC["block_scores"] - 11.48e9) < 0.01e9


def test_block_scores_ceiling():
    # two tensor-core passes over the same logits against one counted contraction
    assert bench.ALGORITHMIC_CEILING == {"block_scores": 0.5}
