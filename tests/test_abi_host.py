"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, rejects bad arguments on the host before touching CUDA,
and plans as the shared-memory budget dictates."""
import ctypes
import json
import os
import re

import pytest

from tiled_staged_matmul_gb300.csrc import build as tsm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsm_gemm.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def b():
    tsm_build.build()
    from tiled_staged_matmul_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(gemm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gemm_f16_f32acc", "gemm_f16_f32acc_batched", "gemm_get_device_status",
              "gemm_last_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(b):
    lib = ctypes.CDLL(b.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_names(b):
    assert b.gemm_version() >= 100
    assert b.gemm_status_string(b.GEMM_ERR_ALIAS) == "GEMM_ERR_ALIAS"
    assert b.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


# Fake, never-dereferenced device addresses: every case below is rejected by
# the host-side checks before any CUDA call is made.
A0, B0, C0 = 0x7f0000000000, 0x7f0010000000, 0x7f0020000000


@pytest.mark.parametrize("args,status", [
    ((A0, B0, 0, 4, 4, 4, 8, 8, 4), "GEMM_ERR_INVALID_VALUE"),        # C NULL
    ((A0, B0, C0, -1, 4, 4, 8, 8, 4), "GEMM_ERR_INVALID_VALUE"),      # negative M
    ((A0, B0, C0, 4, 4, 2**31, 2**31, 8, 4), "GEMM_ERR_INVALID_VALUE"),  # K too large
    ((A0, B0, C0, 4, 4, 16, 8, 8, 4), "GEMM_ERR_INVALID_VALUE"),      # lda < K
    ((A0, B0, C0, 4, 16, 4, 8, 8, 16), "GEMM_ERR_INVALID_VALUE"),     # ldb < N
    ((A0, B0, C0, 4, 8, 4, 8, 8, 4), "GEMM_ERR_INVALID_VALUE"),       # ldc < N
    ((0, B0, C0, 4, 4, 4, 8, 8, 4), "GEMM_ERR_INVALID_VALUE"),        # A NULL
    ((A0 + 1, B0, C0, 4, 4, 4, 8, 8, 4), "GEMM_ERR_MISALIGNED"),      # A: f16 at an odd address
    ((A0, B0 + 3, C0, 4, 4, 4, 8, 8, 4), "GEMM_ERR_MISALIGNED"),      # B: f16 at an odd address
    ((A0, B0, C0 + 2, 4, 4, 4, 8, 8, 4), "GEMM_ERR_MISALIGNED"),      # C: f32 not 4-byte aligned
    ((A0, B0, A0 + 16, 4, 4, 4, 8, 8, 4), "GEMM_ERR_ALIAS"),          # C inside A
    ((A0, B0, B0, 4, 4, 4, 8, 8, 4), "GEMM_ERR_ALIAS"),               # C on B
])
def test_host_rejects_bad_arguments(b, args, status):
    st = b.gemm_f16_f32acc(*args, 0)
    assert b.gemm_status_string(st) == status
    assert b.gemm_last_error_string() != ""


def test_empty_problems_need_no_gpu(b):
    assert b.gemm_f16_f32acc(0, 0, 0, 0, 5, 7, 8, 8, 8, 0) == b.GEMM_OK
    assert b.gemm_f16_f32acc(0, 0, 0, 5, 0, 7, 8, 8, 8, 0) == b.GEMM_OK
    assert b.gemm_f16_f32acc_batched(A0, B0, C0, 4, 4, 4, 8, 8, 4, 0, 0, 0, 0, 0) == b.GEMM_OK


def test_batched_strides_checked(b):
    # overlapping batches of C
    st = b.gemm_f16_f32acc_batched(A0, B0, C0, 4, 4, 4, 8, 8, 4, 32, 32, 8, 2, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_ALIAS"
    # non-positive stride with batch > 1
    st = b.gemm_f16_f32acc_batched(A0, B0, C0, 4, 4, 4, 8, 8, 4, 0, 32, 16, 2, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_INVALID_VALUE"
    # (a stride that is not a multiple of 8 elements is served by repacking:
    # tests/test_gemm_gpu.py covers it on the GPU)


def test_grouped_host_checks(b):
    G0 = 0x7f0030000000
    args = (A0, B0, C0)
    # groups < 0, NULL counts, misaligned counts: rejected on the host
    st = b.gemm_f16_f32acc_grouped(*args, G0, -1, 4, 4, 4, 8, 8, 4, 32, 32, 16, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_INVALID_VALUE"
    st = b.gemm_f16_f32acc_grouped(*args, 0, 2, 4, 4, 4, 8, 8, 4, 32, 32, 16, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_INVALID_VALUE"
    st = b.gemm_f16_f32acc_grouped(*args, G0 + 2, 2, 4, 4, 4, 8, 8, 4, 32, 32, 16, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_MISALIGNED"
    # the batched rules apply per launch (overlapping groups of C)
    st = b.gemm_f16_f32acc_grouped(*args, G0, 2, 4, 4, 4, 8, 8, 4, 32, 32, 8, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_ALIAS"
    # nothing to do: no groups, no rows, no columns
    assert b.gemm_f16_f32acc_grouped(*args, G0, 0, 4, 4, 4, 8, 8, 4, 32, 32, 16, 0) == b.GEMM_OK
    assert b.gemm_f16_f32acc_grouped(*args, G0, 3, 0, 4, 4, 8, 8, 4, 32, 32, 16, 0) == b.GEMM_OK
    assert b.gemm_f16_f32acc_grouped(*args, G0, 3, 4, 0, 4, 8, 8, 8, 32, 32, 16, 0) == b.GEMM_OK


# ---------------------------------------------------------------- planner

SMS = 152


def test_stage_footprint_matches_the_pages_arithmetic(b):
    """The pages stage a 64 x 128 f16 A tile (16384 B) and a 128 x 128 f16 B
    tile (32768 B), 48 KiB in all.  The 128 x 256 x 64 k-block staged here
    holds the same byte counts: a 128 x 64 A tile and a 64 x 256 B tile."""
    g = json.load(open(os.path.join(GOLDEN, "slm_footprint.json")))
    e = g["dtype_bytes"]
    assert g["M"] * g["K"] * e == g["a_tile_bytes"]
    assert g["K"] * g["N"] * e == g["b_tile_bytes"]
    assert g["a_tile_bytes"] + g["b_tile_bytes"] == g["total_bytes"]
    assert (g["total_bytes"] <= g["budget_bytes"]) == g["fits"]
    p = b.gemm_plan(8192, 8192, 8192, 1, b._opts(tile_n=256, tile_m=128), SMS)
    assert p["tile_m"] * p["tile_k"] * e == g["a_tile_bytes"]
    assert p["tile_k"] * p["tile_n"] * e == g["b_tile_bytes"]
    assert p["stage_bytes"] == g["total_bytes"]


@pytest.mark.parametrize("tile_m,tile_n", [(128, 64), (128, 128), (128, 256), (256, 128), (256, 256),
                                           (256, 512)])
def test_ring_fills_the_shared_memory_budget(b, tile_m, tile_n):
    p = b.gemm_plan(4096, 4096, 4096, 1, b._opts(tile_n=tile_n, tile_m=tile_m), SMS)
    assert (p["tile_m"], p["tile_n"]) == (tile_m, tile_n)
    # per CTA: 128 rows of A, and all of the tile's B columns (one CTA) or half (a pair)
    b_cols = tile_n if tile_m == 128 else tile_n // 2
    assert p["stage_bytes"] == 2 * 128 * 64 + 2 * 64 * b_cols
    assert p["stages"] >= 2
    assert p["smem_bytes"] <= 232448
    # one more stage would not fit
    assert p["smem_bytes"] + p["stage_bytes"] > 232448 or p["stages"] == 8
    # one CTA per SM, so the two TMEM accumulators (2 x tile_n columns) never contend
    assert p["smem_bytes"] > 232448 // 2


def test_pair_needs_a_wide_tile(b):
    with pytest.raises(b.GemmError):
        b.gemm_plan(4096, 4096, 4096, 1, b._opts(tile_n=64, tile_m=256), SMS)


@pytest.mark.parametrize("M,N,K,wide", [
    (8192, 8192, 8192, True), (6144, 6144, 6144, True), (3072, 3072, 8192, True),
    (16384, 16384, 4096, True), (4096, 4096, 4096, False), (1000, 1000, 1000, False),
    (256, 256, 65536, False), (12288, 12288, 1024, False), (8192, 4096, 8192, False)])
def test_wide_pair_tile_plans(b, M, N, K, wide):
    # The planner takes 256 x 512 tiles where their fewer operand bytes
    # per flop outweigh the unhidden hand-over of the single accumulator
    # and the coarser waves (long K, whole waves); on request it always does.
    assert (b.gemm_plan(M, N, K, 1, None, SMS)["tile_n"] == 512) == wide
    p = b.gemm_plan(M, N, K, 1, b._opts(tile_n=512), SMS)
    # a CTA pair per 256 x 512 tile, whole tiles only: no K split, no tail
    assert (p["tile_m"], p["tile_n"], p["split_k"], p["tail_split"]) == (256, 512, 1, 0)
    tiles = -(-M // 256) * -(-N // 512)
    assert (p["tiles_m"], p["tiles_n"], p["units"]) == (-(-M // 256), -(-N // 512), tiles)
    assert p["grid"] == 2 * min(tiles, SMS // 2)
    assert p["workspace_bytes"] == 0


@pytest.mark.parametrize("M,N,K,groups", [(4096, 14336, 4096, 8), (512, 1408, 2048, 64),
                                          (8192, 8192, 8192, 1), (300, 700, 50, 300)])
def test_grouped_plan(b, M, N, K, groups):
    # whole tiles whatever the options ask, at most 256 groups per launch,
    # the 512-column tile only on request: otherwise the ordinary plan of
    # one launch's groups with no split and no tail
    for o in (None, b._opts(split_k=4), b.GemmOptions(0, 0, 0, 0, 0, 0, 0, 1)):
        p = b.gemm_plan_grouped(M, N, K, groups, o, SMS)
        assert p["split_k"] == 1 and p["tail_split"] == 0 and p["tile_n"] != 512
        per_launch = min(groups, 256)
        assert p["units"] == per_launch * p["tiles_m"] * p["tiles_n"]
        q = b.gemm_plan(M, N, K, per_launch, b.GemmOptions(1, 0, 0, 0, 0, 0, 0, 2), SMS)
        if q["tile_n"] != 512:
            assert (p["tile_m"], p["tile_n"]) == (q["tile_m"], q["tile_n"])
    assert b.gemm_plan_grouped(M, N, K, groups, b._opts(tile_n=512), SMS)["tile_n"] == 512


@pytest.mark.parametrize("M,N,K,batch", [(1, 1, 1, 1), (200, 300, 64, 1), (256, 512, 64, 3),
                                         (257, 513, 65, 2), (8192, 8192, 8192, 2)])
def test_wide_pair_tile_small_ragged_and_batched_plans(b, M, N, K, batch):
    p = b.gemm_plan(M, N, K, batch, b._opts(tile_n=512), SMS)
    tiles = -(-M // 256) * -(-N // 512) * batch
    assert (p["tile_m"], p["tile_n"], p["split_k"], p["tail_split"]) == (256, 512, 1, 0)
    assert p["units"] == tiles and p["grid"] == 2 * min(tiles, SMS // 2)
    assert (p["stages"], p["stage_bytes"]) == (4, 2 * 128 * 64 + 2 * 64 * 256)
    # the planner's own choice for a batch of the headline shape
    if (M, N, K) == (8192, 8192, 8192):
        assert b.gemm_plan(M, N, K, batch, None, SMS)["tile_n"] == 512


def test_wide_pair_tile_rejects_other_shapes(b):
    for o in (b._opts(tile_n=512, tile_m=128), b._opts(tile_n=512, split_k=2), b._opts(tile_n=384)):
        with pytest.raises(b.GemmError):
            b.gemm_plan(4096, 4096, 4096, 1, o, SMS)
    with pytest.raises(b.GemmError):
        b.gemm_plan(4096, 4096, 4096, 1, b._opts(tile_n=512), 1)


@pytest.mark.parametrize("M,N,K", [(64, 128, 128), (1000, 1000, 1000), (4096, 4096, 4096),
                                   (256, 256, 65536), (8192, 8192, 8192), (1, 1, 1),
                                   (300, 7, 100000), (1, 5000, 64), (2304, 2304, 1024),
                                   (6144, 6144, 6144), (4096, 4096, 512)])
def test_plan_invariants(b, M, N, K):
    p = b.gemm_plan(M, N, K, 1, None, SMS)
    assert p["tile_m"] in (128, 256)
    assert p["tiles_m"] == -(-M // p["tile_m"])
    assert p["tiles_n"] == -(-N // p["tile_n"])
    assert p["k_blocks"] == -(-K // 64)
    assert 1 <= p["split_k"] <= p["k_blocks"]
    tiles = p["tiles_m"] * p["tiles_n"]
    if p["tail_split"]:
        # split tail: whole tiles for the full waves, the rest split tail_split
        # ways -- K ranges summed in the kernel, or column slices of at least
        # 64 B columns per CTA with no partial sums
        slots = SMS // (2 if p["tile_m"] == 256 else 1)
        assert p["split_k"] == 1 and bool(p["fused_reduce"]) != bool(p["tail_narrow"])
        assert p["tail_tiles"] == tiles % slots and p["tail_split"] >= 2
        if p["tail_narrow"]:
            b_cols = p["tile_n"] // (2 if p["tile_m"] == 256 else 1)
            assert p["tail_split"] in (2, 4) and b_cols // p["tail_split"] >= 64
        assert p["units"] == tiles - p["tail_tiles"] + p["tail_tiles"] * p["tail_split"]
        assert p["tail_tiles"] * p["tail_split"] <= slots
    else:
        assert p["units"] == tiles * p["split_k"]
    if p["tile_m"] == 128:
        assert p["grid"] == min(p["units"], SMS)
        assert p["red_cluster"] in (1, 2, 4)
    else:
        assert p["grid"] == 2 * min(p["units"], SMS // 2)
    ldw = -(-N // 4) * 4
    tile_bytes = p["tile_m"] * p["tile_n"] * 4
    if p["tail_narrow"]:
        assert p["workspace_bytes"] == 0
    elif p["tail_split"]:
        counters = -(-(p["tail_tiles"] * 4) // 16) * 16 + 16  # + launch tag
        assert p["workspace_bytes"] == p["tail_tiles"] * p["tail_split"] * tile_bytes + counters
    elif p["split_k"] == 1:
        assert p["workspace_bytes"] == 0 and not p["fused_reduce"]
    elif p["fused_reduce"] and p["red_cluster"] > 1:
        # cluster sum: one compact partial tile per cluster (none with one
        # cluster per tile), one arrival counter per tile and cluster rank
        cl = p["red_cluster"]
        assert p["tile_m"] == 128 and p["split_k"] % cl == 0 and p["grid"] % cl == 0
        groups = p["split_k"] // cl
        counters = -(-(tiles * cl * 4) // 16) * 16 + 16  # + launch tag
        assert p["workspace_bytes"] == tiles * (groups if groups > 1 else 0) * tile_bytes + counters
        assert p["units"] == p["grid"] and p["grid"] // cl <= (SMS // 4 * 18 // 19 if cl == 4 else SMS // 2)
    elif p["fused_reduce"]:
        # one compact partial tile per split unit, one arrival counter per tile;
        # every cluster owns exactly one unit
        counters = -(-(tiles * 4) // 16) * 16 + 16  # + launch tag
        assert p["workspace_bytes"] == tiles * p["split_k"] * tile_bytes + counters
        assert p["units"] * (2 if p["tile_m"] == 256 else 1) == p["grid"]
    else:
        assert p["workspace_bytes"] == p["split_k"] * M * ldw * 4


def test_long_K_small_output_splits_K(b):
    p = b.gemm_plan(256, 256, 65536, 1, None, SMS)
    assert p["split_k"] > 1
    assert p["grid"] <= SMS
    assert p["k_blocks"] // p["split_k"] >= 4


def test_large_square_uses_wide_tiles_without_split(b):
    p = b.gemm_plan(8192, 8192, 8192, 1, None, SMS)
    assert (p["tile_m"], p["tile_n"], p["split_k"]) == (256, 512, 1)  # CTA pairs


def cluster_opts(b, red_cluster, split_k=0, tile_n=0):
    o = b.GemmOptions()
    o.split_k = split_k
    o.red_cluster = red_cluster
    if tile_n:
        o.tile_m, o.tile_n = 128, tile_n
    return o


def test_long_K_small_output_sums_in_clusters_on_request(b):
    # off unless asked for (measured slower than the split-by-split sum)
    p = b.gemm_plan(256, 256, 65536, 1, None, SMS)
    assert (p["tile_m"], p["tile_n"], p["red_cluster"], p["split_k"], p["grid"]) == (128, 128, 1, 38, 152)
    # four 128 x 128 tiles; 36 four-CTA clusters fit on 152 SMs (the GPCs'
    # SMs past a multiple of four stay idle): 9 clusters per tile, 36 K ranges
    p = b.gemm_plan(256, 256, 65536, 1, cluster_opts(b, 4), SMS)
    assert (p["tile_m"], p["tile_n"], p["red_cluster"], p["split_k"], p["grid"]) == (128, 128, 4, 36, 144)
    # pairs: 76 clusters, 19 per tile
    p = b.gemm_plan(256, 256, 65536, 1, cluster_opts(b, 2), SMS)
    assert (p["red_cluster"], p["split_k"], p["grid"]) == (2, 38, 152)
    # off: one partial per K range, as before
    p = b.gemm_plan(256, 256, 65536, 1, cluster_opts(b, 1), SMS)
    assert (p["red_cluster"], p["split_k"], p["grid"]) == (1, 38, 152) and p["fused_reduce"]


def test_cluster_sum_with_a_requested_split(b):
    # a split that is a multiple of the cluster and fits: kept
    p = b.gemm_plan(256, 256, 65536, 1, cluster_opts(b, 4, 16, 128), SMS)
    assert (p["red_cluster"], p["split_k"], p["grid"]) == (4, 16, 64)
    # not a multiple of the cluster: summed split by split
    p = b.gemm_plan(256, 256, 65536, 1, cluster_opts(b, 4, 38, 128), SMS)
    assert (p["red_cluster"], p["split_k"]) == (1, 38)
    # more clusters than fit at once: never (the CTAs wait for one another)
    p = b.gemm_plan(256, 256, 65536, 1, cluster_opts(b, 4, 37 + 3, 128), SMS)
    assert p["red_cluster"] == 1
    # 128 x 256 tiles (two of them): 18 clusters each, 72 K ranges
    p = b.gemm_plan(256, 256, 65536, 1, cluster_opts(b, 4, 0, 256), SMS)
    assert (p["red_cluster"], p["split_k"], p["grid"]) == (4, 72, 144)
    with pytest.raises(b.GemmError):
        b.gemm_plan(256, 256, 65536, 1, cluster_opts(b, 3), SMS)


def test_cluster_sum_of_one_cluster_per_tile(b):
    # 16 k-blocks: one four-CTA cluster per tile holds the whole K (4 ranges
    # of 4 k-blocks) and writes C itself -- no partials in the workspace
    p = b.gemm_plan(128, 128, 1024, 1, cluster_opts(b, 4, 0, 128), SMS)
    assert (p["red_cluster"], p["split_k"]) == (4, 4)
    assert p["workspace_bytes"] == 16 + 16


def test_no_cluster_sum_for_pairs_tails_or_the_separate_reduce(b):
    assert b.gemm_plan(8192, 8192, 8192, 1, cluster_opts(b, 4), SMS)["red_cluster"] == 1
    o = cluster_opts(b, 4)
    o.splitk_reduce = 1
    assert b.gemm_plan(256, 256, 65536, 1, o, SMS)["red_cluster"] == 1
    o = cluster_opts(b, 4)
    o.tile_m, o.tile_n = 256, 256
    assert b.gemm_plan(512, 512, 65536, 1, o, SMS)["red_cluster"] == 1


def test_forced_split_is_clamped_to_k_blocks(b):
    p = b.gemm_plan(128, 128, 128, 1, b._opts(split_k=64), SMS)
    assert p["split_k"] == 2


def test_bad_options_rejected(b):
    with pytest.raises(b.GemmError):
        b.gemm_plan(128, 128, 128, 1, b._opts(tile_n=96), SMS)


def test_separate_reduce_can_be_forced(b):
    p = b.gemm_plan(256, 256, 65536, 1, b._opts(splitk_reduce=1), SMS)
    assert p["split_k"] > 1 and not p["fused_reduce"]
    assert p["workspace_bytes"] == p["split_k"] * 256 * 256 * 4
    with pytest.raises(b.GemmError):
        b.gemm_plan(256, 256, 65536, 1, b._opts(splitk_reduce=3), SMS)


def test_more_units_than_clusters_never_fuses(b):
    # 64 splits of four 128 x 128 tiles = 256 units > 152 CTAs: a CTA would
    # wait on a split that only it can compute later, so the sum is a second kernel.
    p = b.gemm_plan(256, 256, 65536, 1, b._opts(split_k=64, tile_m=128, tile_n=128), SMS)
    assert p["units"] > SMS and not p["fused_reduce"]


def test_split_tail_for_partial_last_waves(b):
    on = b.GemmOptions(0, 0, 0, 0, 0, 0, 0, 1)
    never = b.GemmOptions(0, 0, 0, 0, 0, 0, 0, 2)
    # 1024 pair tiles on 76 clusters: 13 full waves, 36 tiles left, split 2 ways
    p = b.gemm_plan(8192, 8192, 8192, 1, on, SMS)
    assert (p["tail_tiles"], p["tail_split"]) == (36, 2)
    assert p["units"] == 1024 - 36 + 72 and p["fused_reduce"]
    # a last wave more than half full keeps whole tiles
    p = b.gemm_plan(6144, 6144, 6144, 1, on, SMS)
    assert p["tail_split"] == 0 and not p["fused_reduce"]
    # never with the separate-reduce option, nor for batches, nor when asked not to
    off = b.GemmOptions(0, 0, 0, 0, 0, 1, 0, 1)
    assert b.gemm_plan(8192, 8192, 8192, 1, off, SMS)["tail_split"] == 0
    assert b.gemm_plan(4096, 4096, 4096, 2, on, SMS)["tail_split"] == 0
    assert b.gemm_plan(4096, 4096, 4096, 1, never, SMS)["tail_split"] == 0


def test_split_tail_by_default_only_when_it_pays(b):
    def tail(M, N, K, batch=1, opts=None):
        p = b.gemm_plan(M, N, K, batch, opts, SMS)
        return p["tail_split"], "N" if p["tail_narrow"] else ("K" if p["tail_split"] else "-")
    # the planner's choice (options absent or split_tail 0): long enough tiles
    # split in K ranges ...
    assert tail(4096, 4096, 4096) == (2, "K")
    assert tail(8192, 8192, 8192, 1, b._opts(tile_n=256)) == (2, "K")
    assert tail(8192, 8192, 8192) == (0, "-")  # 256 x 512 tiles: whole waves, no tail
    assert tail(2304, 2304, 8192) == (15, "K")
    assert tail(6144, 4096, 4096, 1, b.GemmOptions()) == (16, "K")
    # ... short ones in column slices (storing and summing the partials would
    # cost more than the narrower tiles lose), and batches too
    assert tail(4096, 4096, 1024) == (2, "N")
    assert tail(8192, 8192, 2048) == (2, "N")
    assert tail(8192, 8192, 8192, 3, b._opts(tile_n=256)) == (2, "N")
    # a last wave more than half full stays whole
    assert tail(6144, 6144, 6144) == (0, "-")


def test_column_slice_tail_options(b):
    narrow = b.GemmOptions(0, 0, 0, 0, 0, 0, 0, 3)
    kranges = b.GemmOptions(0, 0, 0, 0, 0, 0, 0, 1)
    # forced either way on 8192^3: 36 tiles left over, halves or two K ranges
    p = b.gemm_plan(8192, 8192, 8192, 1, narrow, SMS)
    assert (p["tail_tiles"], p["tail_split"], p["tail_narrow"]) == (36, 2, 1)
    assert p["units"] == 1024 - 36 + 72 and not p["fused_reduce"] and p["workspace_bytes"] == 0
    p = b.gemm_plan(8192, 8192, 8192, 1, kranges, SMS)
    assert (p["tail_tiles"], p["tail_split"], p["tail_narrow"]) == (36, 2, 0)
    # one CTA per tile: 128 x 256 tiles in quarters when few are left over
    p = b.gemm_plan(1280, 4096, 256, 1, b.GemmOptions(0, 256, 0, 0, 128, 0, 0, 3), SMS)
    assert (p["tail_tiles"], p["tail_split"], p["tail_narrow"]) == (8, 4, 1)
    # a pair tile 128 wide has one 64-column box per CTA: nothing to slice
    p = b.gemm_plan(2304, 2304, 1024, 1, b.GemmOptions(0, 128, 0, 0, 256, 0, 0, 3), SMS)
    assert p["tail_split"] == 0
    # split_tail outside 0..3 is rejected
    with pytest.raises(b.GemmError):
        b.gemm_plan(128, 128, 128, 1, b.GemmOptions(0, 0, 0, 0, 0, 0, 0, 4), SMS)


def test_noalloc_entry_rejects_what_it_cannot_repack(b):
    # host-only: the layout check comes before any CUDA call
    for args in ((A0 + 2, B0, C0, 4, 4, 4, 8, 8, 4), (A0, B0, C0, 4, 4, 4, 12, 8, 4),
                 (A0, B0, C0, 4, 4, 4, 8, 8, 6)):
        st = b.gemm_f16_f32acc_splitk_noalloc(*args, 0, 0)
        assert b.gemm_status_string(st) == "GEMM_ERR_MISALIGNED", args
        assert "cannot repack" in b.gemm_last_error_string()


def test_epilogue_host_checks(b):
    args = (A0, B0, C0, 4, 4, 4, 8, 8, 8, 0, 0, 0, 1)
    bad_act = b.epilogue(activation=9)
    assert b.gemm_status_string(b.gemm_f16_fused(*args, bad_act, None, 0)) == "GEMM_ERR_INVALID_VALUE"
    bad_out = b.epilogue(out_type=7)
    assert b.gemm_status_string(b.gemm_f16_fused(*args, bad_out, None, 0)) == "GEMM_ERR_INVALID_VALUE"
    # a 16-bit C at an odd address, a misaligned bias, a bias overlapping C
    st = b.gemm_f16_fused(A0, B0, C0 + 1, 4, 4, 4, 8, 8, 8, 0, 0, 0, 1, b.epilogue(out_type="bf16"),
                          None, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_MISALIGNED"
    st = b.gemm_f16_fused(*args, b.epilogue(bias=C0 + 0x1000002), None, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_MISALIGNED"
    st = b.gemm_f16_fused(*args, b.epilogue(bias=C0 + 8), None, 0)
    assert b.gemm_status_string(st) == "GEMM_ERR_ALIAS"
    # nothing to do
    assert b.gemm_f16_fused(A0, B0, C0, 0, 4, 4, 8, 8, 8, 0, 0, 0, 1, b.epilogue(activation="gelu"),
                            None, 0) == b.GEMM_OK


def test_rowsum_and_gemv_host_checks(b):
    X0, O0 = 0x7f0040000000, 0x7f0050000000
    bad = lambda st: b.gemm_status_string(st)
    assert bad(b.rowsum_f32acc(X0, 7, O0, 4, 4, 4, 1, 0)) == "GEMM_ERR_INVALID_VALUE"   # element type
    assert bad(b.rowsum_f32acc(X0, "f32", O0, -1, 4, 4, 1, 0)) == "GEMM_ERR_INVALID_VALUE"
    assert bad(b.rowsum_f32acc(X0, "f32", O0, 4, 4, -4, 1, 0)) == "GEMM_ERR_INVALID_VALUE"
    assert bad(b.rowsum_f32acc(X0, "f32", O0, 4, 4, 4, 0, 0)) == "GEMM_ERR_INVALID_VALUE"
    assert bad(b.rowsum_f32acc(X0 + 2, "f32", O0, 4, 4, 4, 1, 0)) == "GEMM_ERR_MISALIGNED"
    assert bad(b.rowsum_f32acc(X0 + 1, "bf16", O0, 4, 4, 4, 1, 0)) == "GEMM_ERR_MISALIGNED"
    assert bad(b.rowsum_f32acc(X0, "f16", X0 + 8, 4, 4, 4, 1, 0)) == "GEMM_ERR_ALIAS"
    assert b.rowsum_f32acc(X0, "f16", O0, 0, 4, 4, 1, 0) == b.GEMM_OK
    assert bad(b.gemv_f16_f32acc(X0, O0, O0 + 64, 4, 8, 4, 1, 0)) == "GEMM_ERR_INVALID_VALUE"  # lda < K
    assert bad(b.gemv_f16_f32acc(X0, O0, X0 + 8, 4, 8, 8, 1, 0)) == "GEMM_ERR_ALIAS"
    assert bad(b.gemv_f16_f32acc(X0, O0 + 1, O0 + 64, 4, 8, 8, 1, 0)) == "GEMM_ERR_MISALIGNED"
    assert b.gemv_f16_f32acc(X0, O0, O0 + 64, 0, 8, 8, 1, 0) == b.GEMM_OK
