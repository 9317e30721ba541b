// gemm_kernel.cuh -- the GEMM kernel template and what it is built from,
// shared by the translation units that instantiate it: gemm_kernels.cu (the
// plain kernels and the cluster split-K sums) and gemm_epi.cu (the kernels
// with a fused epilogue, one unit per activation).  The method and the
// kernel's structure are described at the top of gemm_kernels.cu.
#pragma once

#include "gemm_internal.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tsm {

// ------------------------------------------------------------- tile config

// BN: columns of C per tile.  PAIR: the tile is computed by a CTA pair (a
// 2-CTA cluster) with tcgen05 cta_group::2 -- 256 rows per tile, each CTA
// staging its own 128 rows of A and its own BN/2 columns of B, and holding
// its 128 rows of the accumulator.  Without PAIR one CTA does a 128-row tile.
// A pair's 512-column tile is two 256-column MMAs per k-step on one A tile
// (a quarter fewer operand bytes per flop); its accumulator takes all of
// TMEM, so there is one instead of two.
template <int BN, bool PAIR>
struct TileCfg {
    static_assert(BN == 64 || BN == 128 || BN == 256 || (BN == 512 && PAIR), "tile width");
    static_assert(!PAIR || BN >= 128, "a CTA pair needs at least 64 B columns per CTA");
    static constexpr int ROWS = kTileM;                    // rows of A / C per CTA
    static constexpr int TILE_M = PAIR ? 2 * kTileM : kTileM;
    static constexpr int BK = kTileK;
    static constexpr int B_COLS = PAIR ? BN / 2 : BN;      // B columns staged by one CTA
    static constexpr int A_BYTES = ROWS * BK * 2;          // 16 KiB
    static constexpr int B_BOX_BYTES = 64 * BK * 2;        // one 64-column box: 8 KiB
    static constexpr int B_BOXES = B_COLS / 64;
    static constexpr int B_BYTES = B_BOXES * B_BOX_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // per CTA
    static constexpr int EPI_WARPS = 4;                    // (eight with one buffer each: the same bytes)
    static constexpr int EPI_BUF_BYTES = 32 * 32 * 4;      // one 32 x 32 f32 box
    static constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;
    static constexpr int CTRL_BYTES = 2048;      // barriers and slots, then the group table
    static constexpr int GROUP_TABLE_OFF = 1024; // kMaxGroupsPerLaunch x 4 bytes
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int SMEM_LIMIT = 232448;              // 227 KiB opt-in per block
    static constexpr int STAGES_FIT =
        (SMEM_LIMIT - ALIGN_SLACK - EPI_BYTES - CTRL_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static_assert(STAGES >= 2, "the ring needs at least two stages");
    static_assert(16 * STAGES + 88 <= GROUP_TABLE_OFF &&
                      GROUP_TABLE_OFF + 4 * kMaxGroupsPerLaunch <= CTRL_BYTES,
                  "control block layout");
    static constexpr int SMEM_BYTES = ALIGN_SLACK + STAGES * STAGE_BYTES + EPI_BYTES + CTRL_BYTES;
    // Two accumulators of BN f32 columns each per CTA (a power of two >= 32),
    // or one when two do not fit the 512 TMEM columns.
    static constexpr int ACC = 2 * BN <= 512 ? 2 : 1;
    static constexpr uint32_t TMEM_COLS = uint32_t(ACC * BN);
    // The MMA width: the tile's, in 256-column halves for a 512-column tile.
    static constexpr int MMA_N = BN > 256 ? 256 : BN;
    static constexpr int MMA_HALVES = BN / MMA_N;
    // B boxes of one MMA in a CTA's stage: a pair's MMA takes each CTA's
    // half of its columns, so a 512-column tile's CTA stages, of each
    // 256-column half of the tile, the 128 columns its rank picks.
    static constexpr int B_BOXES_PER_MMA = B_BOXES / MMA_HALVES;
    static_assert(SMEM_BYTES > SMEM_LIMIT / 2, "one CTA per SM keeps TMEM allocation uncontended");
    // Whether the CTA's last unit can stage all its output boxes in the idle
    // ring at once (else it keeps the double-buffered staging).
    static constexpr bool DRAIN_FITS = STAGES * STAGE_BYTES >= EPI_WARPS * (BN / 32) * EPI_BUF_BYTES;
    static_assert(BN == 512 || DRAIN_FITS, "the ring holds a whole output tile of one CTA");
};

// Instruction descriptor of tcgen05.mma.kind::f16: D f32 (bits 4-5 = 1),
// A and B f16 (bits 7-9, 10-12 = 0), A K-major (bit 15 = 0), B MN-major
// (bit 16 = 1: B is row-major K x N, so N is contiguous), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28 (M = 256 for a CTA pair).  N is the MMA's
// width: the tile's, or a column slice of it.
template <int N, bool PAIR>
__device__ __forceinline__ constexpr uint32_t mma_idesc()
{
    static_assert(N % 16 == 0 && N >= 16 && N <= 256, "MMA width");
    return (1u << 4) | (1u << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(PAIR ? 256 : 128) >> 4 << 24);
}

// Shared-memory matrix descriptor fields common to both operands: 128-byte
// swizzle (bits 61-63 = 2), descriptor version 1 (bits 46-48), 8-row groups
// 1024 bytes apart (stride byte offset, bits 32-45, in 16-byte units).
__device__ __forceinline__ uint64_t desc_common()
{
    return (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// A: K-major, one 128-byte row per M row.  The K=16 slice of an MMA lies
// inside one swizzle row, so the leading byte offset is unused (set to 1).
__device__ __forceinline__ uint64_t desc_a(uint32_t saddr)
{
    return desc_common() | (uint64_t(1) << 16) | uint64_t((saddr & 0x3FFFFu) >> 4);
}

// B: MN-major, each 64-column box is K rows of 128 bytes; boxes (64-column
// atoms along N) are 8 KiB apart (leading byte offset).
__device__ __forceinline__ uint64_t desc_b(uint32_t saddr)
{
    return desc_common() | (uint64_t((64 * kTileK * 2) >> 4) << 16) |
           uint64_t((saddr & 0x3FFFFu) >> 4);
}

// ------------------------------------------------------------- helpers

// ------------------------------------------------------------- fused epilogue

// erf(x) by Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: for x >= 0, erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5))))
// e^(-x^2) with t = 1 / (1 + p x), absolute error below 1.5e-7; odd in x.
__device__ __forceinline__ float erf_as(float x)
{
    const float ax = fabsf(x);
    const float t = __fdividef(1.f, fmaf(0.3275911f, ax, 1.f));
    float poly = fmaf(1.061405429f, t, -1.453152027f);
    poly = fmaf(poly, t, 1.421413741f);
    poly = fmaf(poly, t, -0.284496736f);
    poly = fmaf(poly, t, 0.254829592f);
    const float y = 1.f - poly * t * __expf(-ax * ax);
    return copysignf(y, x);
}

// The activations, in f32:
//   relu(v) = v > 0 ? v : 0            leaky_relu(v) = v > 0 ? v : slope v
//   gelu(v) = v/2 (1 + erf(v / sqrt 2))   (erf as above)
//   gelu_tanh(v) = v/2 (1 + tanh u), u = sqrt(2/pi) (v + 0.044715 v^3),
//     tanh u = 1 - 2 / (1 + e^(2u))   (saturates to +-1 for large |u|)
//   silu(v) = v / (1 + e^-v)
// with CUDA's __expf and __fdividef; the errors these add are far below the
// product's own rounding bound.
__device__ __forceinline__ float epi_act(float v, int32_t act, float slope)
{
    switch (act) {
    case kActRelu: return v > 0.f ? v : 0.f;
    case kActLeakyRelu: return v > 0.f ? v : slope * v;
    case kActGelu: return 0.5f * v * (1.f + erf_as(v * 0.70710678118654752f));
    case kActGeluTanh: {
        const float u = 0.79788456080286536f * fmaf(0.044715f * v, v * v, v);
        const float th = 1.f - __fdividef(2.f, 1.f + __expf(2.f * u));
        return 0.5f * v * (1.f + th);
    }
    case kActSilu: return __fdividef(v, 1.f + __expf(-v));
    default: return v;
    }
}

// act(alpha * acc + bias), the value before the output rounding.
__device__ __forceinline__ float epi_value(float acc, float bias, const Epilogue &e)
{
    return epi_act(e.alpha * acc + bias, e.act, e.slope);
}

// An f32 value as the 16-bit output type stores it (round to nearest even).
__device__ __forceinline__ uint32_t epi_out16(float v, int32_t out_type)
{
    return out_type == kOutBF16 ? uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(v)))
                                : uint32_t(__half_as_ushort(__float2half_rn(v)));
}

// An activation as a compile-time constant (template argument of a lambda).
template <int A>
struct ActTag {
    static constexpr int value = A;
};

// The activation of a kernel built for one (ACT >= 0), or read at run time
// (kActRuntime: the cluster split-K sums), as an ActTag for `fn`.
constexpr int kActRuntime = -1;
template <int ACT, typename F>
__device__ __forceinline__ void with_activation(int32_t act, F &&fn)
{
    if constexpr (ACT != kActRuntime) {
        fn(ActTag<ACT>{});
    } else {
        switch (act) {
        case kActRelu: fn(ActTag<kActRelu>{}); break;
        case kActLeakyRelu: fn(ActTag<kActLeakyRelu>{}); break;
        case kActGelu: fn(ActTag<kActGelu>{}); break;
        case kActGeluTanh: fn(ActTag<kActGeluTanh>{}); break;
        case kActSilu: fn(ActTag<kActSilu>{}); break;
        default: fn(ActTag<kActNone>{}); break;
        }
    }
}

// The fused epilogue on four consecutive values of one row (columns col ...
// col + 3), the activation fixed at compile time so that the four overlap:
// v = act(alpha * v + bias[col]).
template <int ACT>
__device__ __forceinline__ void epi_apply4_as(float4 &v, int32_t col, int32_t N, const float *bias,
                                              const Epilogue &e)
{
    float b[4] = {0.f, 0.f, 0.f, 0.f};
    if (bias) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            b[k] = col + k < N ? __ldg(bias + col + k) : 0.f;
    }
    v.x = epi_act(fmaf(e.alpha, v.x, b[0]), ACT, e.slope);
    v.y = epi_act(fmaf(e.alpha, v.y, b[1]), ACT, e.slope);
    v.z = epi_act(fmaf(e.alpha, v.z, b[2]), ACT, e.slope);
    v.w = epi_act(fmaf(e.alpha, v.w, b[3]), ACT, e.slope);
}

// Store one epilogue value at element `idx` of C (f32 or 16-bit).
__device__ __forceinline__ void epi_store(void *C, int64_t idx, float v, int32_t out_type)
{
    if (out_type == kOutF32)
        static_cast<float *>(C)[idx] = v;
    else
        static_cast<uint16_t *>(C)[idx] = uint16_t(epi_out16(v, out_type));
}

struct Unit {
    int32_t m0, n0;    // first row / column of the tile
    int32_t z_in;      // batch index of A and B
    int32_t z_out;     // third coordinate of the output (or workspace) map
    int32_t kb0, kb1;  // k-block range [kb0, kb1)
    int32_t split;     // fused split unit: 1 (its partial goes to the workspace), else 0
    int32_t s;         // fused split unit: its split index
    int64_t red_tile;  // fused split unit: index of its tile among the split tiles
    int32_t rows;      // rows of the matrix: M, or the group's count in a grouped launch
    int32_t width;     // columns of the unit: the tile width, or a slice of it (narrow tail)
};

// Tile index (within one matrix) -> first row / column, in a grouped raster:
// group_m rows of tiles are walked column by column, so CTAs running at the
// same time share A and B panels in L2 ("Intel XPU Backend for Triton",
// section "Use Proper Type Annotations": GROUP_SIZE_M in the GEMM signature).
__device__ __forceinline__ void raster(int64_t t, const KernelParams &p, int32_t tiles_m, int tile_m,
                                       int bn, int32_t &m0, int32_t &n0)
{
    const int64_t group = int64_t(p.group_m) * p.tiles_n;
    const int64_t g = t / group;
    const int32_t first_m = int32_t(g * p.group_m);
    const int32_t rows_in_group = min(tiles_m - first_m, p.group_m);
    const int64_t r = t - g * group;
    m0 = (first_m + int32_t(r % rows_in_group)) * tile_m;
    n0 = int32_t(r / rows_in_group) * bn;
}

// Work unit -> tile and K range.
//   fused plans: units below dp_units are whole tiles; the others are split
//     units, tile-major (the splits of one tile sit on neighbouring clusters);
//     with split_first the split units come first and the whole tiles after.
//   narrow tails: units below dp_units are whole tiles; the others are column
//     slices of the remaining tiles (`narrow` slices of bn / narrow columns
//     each, full K), tile-major.
//   grouped launches: the group whose tiles hold u (binary search of `gtab`,
//     the inclusive tile counts per group), then its tiles as in one matrix.
//   otherwise: (batch, split) outermost, then the tiles of one matrix; split
//     partials go to [batch * split_k + s][M][ldw] for the reduce kernel.
__device__ __forceinline__ Unit decode_unit(int64_t u, const KernelParams &p, const uint32_t *gtab,
                                            int tile_m, int bn)
{
    const int64_t tiles = int64_t(p.tiles_m) * p.tiles_n;
    Unit w;
    w.split = 0;
    w.s = 0;
    w.red_tile = 0;
    w.rows = p.M;
    w.width = bn;
    if (p.group_rows) {
        int32_t lo = 0, hi = p.groups - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi) >> 1;
            if (int64_t(gtab[mid]) > u)
                hi = mid;
            else
                lo = mid + 1;
        }
        const int64_t first = lo ? int64_t(gtab[lo - 1]) : 0;
        const int32_t tiles_m = int32_t((int64_t(gtab[lo]) - first) / p.tiles_n);
        raster(u - first, p, tiles_m, tile_m, bn, w.m0, w.n0);
        w.z_in = lo;
        w.z_out = lo;
        w.kb0 = 0;
        w.kb1 = p.k_blocks;
        w.rows = min(max(p.group_rows[lo], 0), p.M);
        return w;
    }
    if (p.fused || p.narrow) {
        int64_t tg = u;  // tile index over all matrices of the batch
        int32_t piece = 0;
        w.kb0 = 0;
        w.kb1 = p.k_blocks;
        if (p.split_first && u >= p.n_first) {
            tg = u - p.n_first;
        } else if (p.split_first || u >= p.dp_units) {
            const int64_t j = p.split_first ? u : u - p.dp_units;
            const int32_t per = p.narrow ? p.narrow : p.split_k;
            const int64_t t = j / per;
            const int32_t s = int32_t(j - t * per);
            tg = p.dp_units + t;
            if (p.narrow) {
                piece = s;
                w.width = bn / p.narrow;
            } else {
                w.red_tile = t;
                w.s = s;
                w.split = 1;
                w.kb0 = int32_t(int64_t(s) * p.k_blocks / p.split_k);
                w.kb1 = int32_t(int64_t(s + 1) * p.k_blocks / p.split_k);
            }
        }
        const int64_t b = tg / tiles;
        raster(tg - b * tiles, p, p.tiles_m, tile_m, bn, w.m0, w.n0);
        w.n0 += piece * w.width;
        w.z_in = int32_t(b);
        w.z_out = w.split ? int32_t(p.split_first ? u : u - p.dp_units) : int32_t(b);
        return w;
    }
    const int64_t z = u / tiles;
    const int64_t t = u - z * tiles;
    const int32_t b = int32_t(z / p.split_k);
    const int32_t s = int32_t(z - int64_t(b) * p.split_k);
    raster(t, p, p.tiles_m, tile_m, bn, w.m0, w.n0);
    w.z_in = b;
    w.z_out = int32_t(z);  // == b when split_k == 1
    w.kb0 = int32_t(int64_t(s) * p.k_blocks / p.split_k);
    w.kb1 = int32_t(int64_t(s + 1) * p.k_blocks / p.split_k);
    return w;
}

// Where a CTA records that it gives up: its own abort flag and, in a CTA
// pair, the peer's (a shared::cluster address), so that both wind down.
struct AbortFlags {
    volatile uint32_t *local;
    uint32_t peer;       // shared::cluster address of the peer's flag (0: none)
    uint64_t timeout_ns;
    uint32_t *status;
};

// Bounded mbarrier wait.  Returns false if the CTA's abort flag is raised
// (when `honor_abort`) or if `timeout_ns` passes; a timeout raises the flags
// and ORs `who` into the device status word.  CLUSTER_ACQ: the wait acquires
// at cluster scope (for data other CTAs of the cluster counted on `bar`).
template <bool CLUSTER_ACQ = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const AbortFlags &af,
                                             uint32_t who, bool honor_abort)
{
    auto try_wait = [&]() {
        return CLUSTER_ACQ ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (try_wait())
        return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (try_wait())
            return true;
        if ((it & 31u) == 0) {
            if (honor_abort && *af.local)
                return false;
            if (ptx::globaltimer_ns() - t0 > af.timeout_ns) {
                *af.local = 1u;
                if (af.peer)
                    ptx::st_cluster_u32(af.peer, 1u);
                atomicOr(af.status, who);
                return false;
            }
        }
    }
}

// Bounded poll of a global word (acquire, GPU scope) until it equals `want`.
// Returns false if the CTA's abort flag is raised or `timeout_ns` passes; a
// timeout raises the flags and ORs `who` into the device status word.  Every
// waiter polls the same word, so each poll backs off first.
template <typename T>
__device__ __forceinline__ bool poll_bounded(const T *word, T want, const AbortFlags &af,
                                             uint32_t who)
{
    auto load = [word]() -> T {
        if constexpr (sizeof(T) == 8)
            return T(ptx::ld_acquire_gpu(reinterpret_cast<const unsigned long long *>(word)));
        else
            return T(ptx::ld_acquire_gpu_u32(reinterpret_cast<const uint32_t *>(word)));
    };
    if (load() == want)
        return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(64);
        if (load() == want)
            return true;
        if ((it & 7u) == 0) {
            if (*af.local)
                return false;
            if (ptx::globaltimer_ns() - t0 > af.timeout_ns) {
                *af.local = 1u;
                if (af.peer)
                    ptx::st_cluster_u32(af.peer, 1u);
                atomicOr(af.status, who);
                return false;
            }
        }
    }
}

// Grouped launch, run by the 32 lanes of one warp before the CTA barrier:
// table[g] = the number of tiles of groups 0..g, each group having
// ceil(rows / tile_m) x tiles_n tiles for its row count clamped to [0, M]
// (a count outside that range raises kStatusGroupRows).  The prefix is an
// inclusive scan: eight groups per lane, then the lanes' sums by shuffles.
static __device__ __noinline__ void build_group_table(const int32_t *group_rows, int32_t groups, int32_t M,
                                               int32_t tile_m, int32_t tiles_n, uint32_t *table,
                                               uint32_t *status)
{
    constexpr int PER = kMaxGroupsPerLaunch / 32;
    const int lane = int(threadIdx.x & 31);
    uint32_t incl[PER];
    uint32_t sum = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int g = lane * PER + i;
        if (g < groups) {
            int64_t r = group_rows[g];
            if (r < 0 || r > M) {
                bad = true;
                r = r < 0 ? 0 : M;
            }
            sum += uint32_t((r + tile_m - 1) / tile_m) * uint32_t(tiles_n);
        }
        incl[i] = sum;
    }
    uint32_t scan = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, scan, d);
        if (lane >= d)
            scan += v;
    }
    const uint32_t before = scan - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i)
        if (lane * PER + i < groups)
            table[lane * PER + i] = before + incl[i];
    if (bad)
        atomicOr(status, kStatusGroupRows);
}

// In-kernel split-K, run by one thread of CTA 0 at the start: zero this
// launch's arrival counters, then publish the launch's epoch.  Kept out of
// line: the kernels that do not sum in-kernel only pay for the call site.
static __device__ __noinline__ void publish_counters(uint32_t *counters, int32_t words,
                                              unsigned long long *tag, uint64_t epoch)
{
    for (int32_t i = 0; i < words; ++i)
        counters[i] = 0u;
    __threadfence();
    ptx::st_release_gpu(tag, epoch);
}

__device__ __forceinline__ void trace_stamp(const KernelParams &p, int slot)
{
    if (p.trace)
        p.trace[int64_t(blockIdx.x) * kTraceSlots + slot] = ptx::globaltimer_ns();
}

// ------------------------------------------------------------- cluster split-K sum

// The epilogue of the cluster split-K sum (warps 2..5; one split unit per
// CTA, clusters of CL = p.red_cluster CTAs holding CL consecutive K ranges
// of one 128-row tile, every CTA of the launch resident at once).
//
//  1. Once its accumulator is complete, every MMA that read the CTA's operand
//     ring has finished, so the ring is idle: the CTA tells its peers so.
//  2. CTA rank r owns tile rows [r * 128 / CL, (r + 1) * 128 / CL).  Each
//     epilogue warp reads its 32 TMEM rows box by box (32 x 32 f32, in the
//     128-byte swizzled layout of the C boxes): an owner's own rows go into
//     its slot for its own rank; other rows are staged in the idle ring past
//     the slots and sent to the owner's slot for this rank with one bulk copy
//     per box (cp.async.bulk into distributed shared memory), counted on the
//     owner's recv_full.
//  3. The owner adds its CL slots in ascending rank (= split) order.  With one
//     cluster per tile that is C (through the epilogue); otherwise the sum is
//     TMA-stored to the workspace as cluster partial g and the tile's G
//     cluster partials of the owner's rows are summed in ascending g, rows_per
//     rows per CTA, after every CTA holding those rows has arrived -- the
//     same arrival, load and sum as the plain in-kernel split-K sum.
// Shared memory: [0, CL x slot) the receive slots (later the target of the
// load of the cluster partials), then (CL - 1) x slot of outgoing staging;
// the planner checks that both fit the ring and the epilogue buffers.
template <int BN, bool EPI>
__device__ __forceinline__ void cluster_sum_epilogue(
    const KernelParams &p, const CUtensorMap &map_ws, const CUtensorMap &map_red, uint32_t base,
    uint8_t *base_ptr, uint32_t tmem_base, uint32_t tfull0, uint32_t stall_bar, uint32_t red_bar,
    uint32_t peers_free, uint32_t recv_full, volatile uint32_t *red_ok, volatile uint32_t *clu_bad,
    volatile uint32_t *abort_flag, const AbortFlags &af, int64_t num_units, int warp, int lane)
{
    using Cfg = TileCfg<BN, false>;
    constexpr uint32_t BOX = Cfg::EPI_BUF_BYTES;  // one 32 x 32 f32 box
    const int q = warp & 3;                       // TMEM lanes 32q ... 32q + 31 = tile rows
    const int et = int(threadIdx.x) - 64;         // 0..127
    if (blockIdx.x == 0 && threadIdx.x == 64)
        publish_counters(p.counters, p.counter_words, p.epoch_tag, p.epoch);
    const int CL = p.red_cluster;
    const int G = p.red_groups;
    const uint32_t crank = ptx::cluster_ctarank();
    const int per = 4 / CL;                       // epilogue warps whose rows one CTA owns
    const int rows_own = Cfg::ROWS / CL;
    const int32_t own0 = int32_t(crank) * rows_own;
    const uint32_t slot_bytes = uint32_t(rows_own) * BN * 4u;
    const bool has_unit = int64_t(blockIdx.x) < num_units;
    const Unit w = has_unit ? decode_unit(blockIdx.x, p, nullptr, Cfg::TILE_M, BN) : Unit{};
    const int g = w.s / CL;

    bool ok = has_unit && uint32_t(w.s % CL) == crank;
    ok = ok && wait_bounded(tfull0, 0, af, kStatusEpilogue, true);
    if (p.inject_stall && ok)
        ok = wait_bounded(stall_bar, 0, af, kStatusEpilogue, true);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after_sync();
    if (warp == 2 && lane == 0)
        trace_stamp(p, kTraceAccReady);
    // 1.  (The wait on the setup arrive makes sure the peers' barriers exist.)
    ptx::cluster_wait();
    if (ok && warp == 2 && lane == 0) {
        for (int r = 0; r < CL; ++r)
            if (r != int(crank))
                ptx::mbar_arrive_cluster(ptx::mapa_shared(peers_free, uint32_t(r)));
    }
    // 2.
    const int owner = q / per;
    const bool local = owner == int(crank);
    const uint32_t slot = base + crank * slot_bytes + uint32_t(q - owner * per) * uint32_t(BN / 32) * BOX;
    const int sidx = q < int(crank) * per ? q : q - per;  // index among this CTA's sending warps
    const uint32_t stage = base + uint32_t(CL) * slot_bytes + uint32_t(sidx) * uint32_t(BN / 32) * BOX;
    if (ok && !local)
        ok = wait_bounded(peers_free, 0, af, kStatusReduce, true);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
        const uint32_t bar = ptx::mapa_shared(recv_full, uint32_t(owner));
        const uint32_t tm_row = tmem_base + (uint32_t(32 * q) << 16);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(tm_row + 32u * uint32_t(c), r);
            ptx::tmem_wait_ld();
            const uint32_t buf = (local ? slot : stage) + uint32_t(c) * BOX;
            const uint32_t row_addr = buf + uint32_t(lane) * 128u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ptx::st_shared_v4(row_addr + (uint32_t(j ^ (lane & 7)) << 4), r[4 * j], r[4 * j + 1],
                                  r[4 * j + 2], r[4 * j + 3]);
            if (!local) {
                ptx::fence_proxy_async_smem();  // the box before the bulk copy reads it
                __syncwarp();
                if (lane == 0)
                    ptx::bulk_copy_to_cluster(ptx::mapa_shared(slot + uint32_t(c) * BOX, uint32_t(owner)),
                                              buf, BOX, bar);
            }
        }
    }
    // The owned rows: the peers' (counted on recv_full, acquired at cluster
    // scope) and this CTA's own warps' (the named barrier).
    if (ok)
        ok = wait_bounded<true>(recv_full, 0, af, kStatusReduce, true);
    if (!ok)
        *clu_bad = 1u;
    ptx::named_bar_sync(1, 128);
    const bool go = *clu_bad == 0u;

    // Four sums of one row of the tile (tile row tr, columns tc ... tc + 3)
    // through the epilogue into C, clipped at M and N.
    auto put4 = [&](auto act, int32_t tr, int32_t tc, const float4 &acc) {
        const int32_t gr = w.m0 + tr;
        const int32_t gc = w.n0 + tc;
        if (gr >= p.M || gc >= p.N)
            return;
        const int64_t bz = w.z_in;
        const int64_t at = bz * p.stride_c + int64_t(gr) * p.ldc + gc;
        if constexpr (EPI) {
            const float *bias = p.epi.bias ? p.epi.bias + bz * p.epi.bias_stride : nullptr;
            float4 v = acc;
            epi_apply4_as<decltype(act)::value>(v, gc, p.N, bias, p.epi);
            if (gc + 3 < p.N && p.epi.out_type == kOutF32) {
                *reinterpret_cast<float4 *>(static_cast<float *>(p.c_direct) + at) = v;
            } else if (gc + 3 < p.N) {
                *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.c_direct) + at) =
                    make_uint2(epi_out16(v.x, p.epi.out_type) | (epi_out16(v.y, p.epi.out_type) << 16),
                               epi_out16(v.z, p.epi.out_type) | (epi_out16(v.w, p.epi.out_type) << 16));
            } else {
                const float vv[3] = {v.x, v.y, v.z};
#pragma unroll
                for (int k = 0; k < 3; ++k)
                    if (gc + k < p.N)
                        epi_store(p.c_direct, at + k, vv[k], p.epi.out_type);
            }
        } else {
            float *dst = static_cast<float *>(p.c_direct) + at;
            if (gc + 3 < p.N) {
                *reinterpret_cast<float4 *>(dst) = acc;
            } else {
                dst[0] = acc.x;
                if (gc + 1 < p.N)
                    dst[1] = acc.y;
                if (gc + 2 < p.N)
                    dst[2] = acc.z;
            }
        }
    };
    auto with_act = [&](auto &&fn) {
        if constexpr (EPI) {
            switch (p.epi.act) {
            case kActRelu: fn(ActTag<kActRelu>{}); break;
            case kActLeakyRelu: fn(ActTag<kActLeakyRelu>{}); break;
            case kActGelu: fn(ActTag<kActGelu>{}); break;
            case kActGeluTanh: fn(ActTag<kActGeluTanh>{}); break;
            case kActSilu: fn(ActTag<kActSilu>{}); break;
            default: fn(ActTag<kActNone>{}); break;
            }
        } else {
            fn(ActTag<kActNone>{});
        }
    };

    // 3.  Chunk f (16 bytes) of a slot: box f / 256 (row block, then column
    // box), row (f / 8) % 32, column chunk (f % 8) ^ row % 8.
    const int nf = rows_own * BN / 4;
    float4 *const slots = reinterpret_cast<float4 *>(base_ptr);
    if (go) {
        with_act([&](auto act) {
            for (int f = et; f < nf; f += 128) {
                float4 a = slots[f];
                for (int r = 1; r < CL; ++r) {
                    const float4 v = slots[r * nf + f];
                    a.x += v.x;
                    a.y += v.y;
                    a.z += v.z;
                    a.w += v.w;
                }
                if (G == 1) {
                    const int bx = f >> 8, i = (f >> 3) & 31, j = (f & 7) ^ (i & 7);
                    put4(act, own0 + 32 * (bx / (BN / 32)) + i, 32 * (bx % (BN / 32)) + 4 * j, a);
                } else {
                    slots[f] = a;
                }
            }
        });
    }
    if (G == 1) {
        ptx::named_bar_sync(1, 128);
        if (et == 0)
            trace_stamp(p, kTraceReduced);
        return;
    }
    // The cluster partial of the owned rows to the workspace.
    ptx::fence_proxy_async_smem();  // the sums above before the TMA store reads them
    ptx::named_bar_sync(1, 128);
    uint64_t epoch_now = 0;
    if (et == 0) {
        epoch_now = ptx::ld_relaxed_gpu(p.epoch_tag);
        if (go) {
            for (int rb = 0; rb < rows_own / 32; ++rb)
                for (int cb = 0; cb < BN / 32; ++cb)
                    ptx::tma_store_3d(&map_ws, base + uint32_t(rb * (BN / 32) + cb) * BOX, 32 * cb,
                                      own0 + 32 * rb, int32_t(w.red_tile * G + g));
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_all();
            ptx::fence_proxy_async_global();
        }
        trace_stamp(p, kTraceStored);
    }
    // Arrive on the (tile, rank) counter once the partial is in the
    // workspace, wait (bounded) for the tile's G clusters, fetch rows
    // [r0, r0 + rows_per) of the G partials with one TMA load into the slots
    // (summed and stored above: free again), add them in ascending g.
    const int32_t r0 = own0 + g * p.rows_per;
    const bool active = g * p.rows_per < rows_own && w.m0 + r0 < p.M;
    if (et == 0) {
        uint32_t okv = 0;
        if (go) {
            const bool epoch_ok = epoch_now == p.epoch ||
                poll_bounded<unsigned long long>(p.epoch_tag, p.epoch, af, kStatusReduce);
            if (!*abort_flag && epoch_ok) {
                uint32_t *count = p.counters + w.red_tile * CL + crank;
                __threadfence();
                atomicAdd(count, 1u);  // arrive
                okv = poll_bounded<uint32_t>(count, uint32_t(G), af, kStatusReduce);
                if (okv && active) {
                    ptx::fence_proxy_async_global();
                    ptx::mbar_arrive_expect_tx(red_bar, uint32_t(p.rows_per) * BN * 4u * uint32_t(G));
                    ptx::tma_load_3d(base, &map_red, red_bar, 0, r0, int32_t(w.red_tile * G));
                }
            }
        }
        *red_ok = okv;
    }
    ptx::named_bar_sync(1, 128);
    if (*red_ok && active && wait_bounded(red_bar, 0, af, kStatusReduce, false)) {
        const int32_t per_split = p.rows_per * (BN / 4);  // float4s of one cluster partial
        const int32_t row_end = own0 + rows_own;
        with_act([&](auto act) {
            for (int32_t f = et; f < per_split; f += 128) {
                float4 a = slots[f];
#pragma unroll 4
                for (int32_t s2 = 1; s2 < G; ++s2) {
                    const float4 v = slots[s2 * per_split + f];
                    a.x += v.x;
                    a.y += v.y;
                    a.z += v.z;
                    a.w += v.w;
                }
                const int32_t row = f / (BN / 4);
                if (r0 + row < row_end)
                    put4(act, r0 + row, (f - row * (BN / 4)) * 4, a);
            }
        });
    }
    ptx::named_bar_sync(1, 128);
    if (et == 0)
        trace_stamp(p, kTraceReduced);
}

// ------------------------------------------------------------- the GEMM

// ACT: the fused epilogue's activation (kActNone in the plain kernels;
// kActRuntime: read from p.epi.act).
template <int BN, bool PAIR, bool EPI, bool CLU, int ACT>
__global__ void __launch_bounds__(gemm_threads(EPI, CLU), 1)
    tsm_gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap map_a,
                            const __grid_constant__ CUtensorMap map_b,
                            const __grid_constant__ CUtensorMap map_out,
                            const __grid_constant__ CUtensorMap map_ws,
                            const __grid_constant__ CUtensorMap map_red, const KernelParams p)
{
    using Cfg = TileCfg<BN, PAIR>;
    constexpr int S = Cfg::STAGES;
    static_assert(!(CLU && PAIR), "the cluster split-K sum is built for one CTA per tile");
    // Epilogue warps: four (one per TMEM lane quarter), or with a fused
    // epilogue eight -- two per quarter, taking alternate boxes of its rows,
    // so that one warp's arithmetic latency hides behind the other's (a
    // single warp per sub-partition issues well below one instruction per
    // cycle on the activation's dependent chains).  The staging space stays
    // the same: one box buffer per warp instead of two.
    constexpr int EW = epilogue_warps(EPI, CLU);
    constexpr int HW = EW / 4;   // epilogue warps per TMEM lane quarter
    constexpr int ET = 32 * EW;  // epilogue threads
    constexpr int NBUF = 2 / HW; // staging buffers per epilogue warp
    static_assert(EW * NBUF * Cfg::EPI_BUF_BYTES == Cfg::EPI_BYTES, "epilogue staging");
    constexpr uint32_t TEMPTY = uint32_t((PAIR ? 2 : 1) * EW);  // arrivals that free an accumulator

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 B
    uint8_t *const base_ptr = smem_raw + (base - raw);
    const uint32_t epi0 = base + S * Cfg::STAGE_BYTES;
    const uint32_t ctrl = epi0 + Cfg::EPI_BYTES;
    uint8_t *const ctrl_ptr = base_ptr + (ctrl - base);

    // Control block: barriers (8 bytes each), then the TMEM address and the
    // CTA's abort flag.  In a CTA pair `full` and `tempty` are used in the
    // leader only; `empty` and `tfull` in both (the leader's MMA commits
    // arrive on both CTAs' copies).
    const uint32_t full0 = ctrl;                     // [S]  TMA bytes landed in slot s
    const uint32_t empty0 = ctrl + 8u * S;           // [S]  MMAs reading slot s are done
    const uint32_t tfull0 = ctrl + 16u * S;          // [2]  accumulator b is complete
    const uint32_t tempty0 = ctrl + 16u * S + 16u;   // [2]  epilogue has read accumulator b
    const uint32_t done_bar = ctrl + 16u * S + 32u;  // all MMAs of this CTA (pair) completed
    const uint32_t stall_bar = ctrl + 16u * S + 40u; // never signalled (test hook)
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(ctrl_ptr + 16 * S + 48);
    uint32_t *const gtab = reinterpret_cast<uint32_t *>(ctrl_ptr + Cfg::GROUP_TABLE_OFF);
    volatile uint32_t *const abort_flag = tmem_slot + 1;
    volatile uint32_t *const red_ok = tmem_slot + 2;  // in-kernel split-K: go / no-go
    const uint32_t red_bar = ctrl + 16u * S + 64u;    // in-kernel split-K: partial chunks landed
    volatile uint32_t *const clu_bad = tmem_slot + 3; // cluster sum: some epilogue warp gave up
    const uint32_t peers_free = ctrl + 16u * S + 72u; // cluster sum: every peer's ring is idle
    const uint32_t recv_full = ctrl + 16u * S + 80u;  // cluster sum: the peers' rows have landed

    const int warp = int(threadIdx.x >> 5);
    const int lane = int(threadIdx.x & 31);
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;  // 0: the pair's MMA issuer
    const bool leader = rank == 0;
    const int64_t cluster = PAIR ? (blockIdx.x >> 1) : blockIdx.x;
    const int64_t nclusters = PAIR ? (gridDim.x >> 1) : gridDim.x;

    if (threadIdx.x == 0) {
        trace_stamp(p, kTraceEntry);
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full0 + 8u * s, 1);
            ptx::mbar_init(empty0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull0 + 8u * b, 1);
            ptx::mbar_init(tempty0 + 8u * b, TEMPTY);
        }
        ptx::mbar_init(done_bar, 1);
        ptx::mbar_init(stall_bar, 1);
        ptx::mbar_init(red_bar, 1);
        *abort_flag = 0u;
        if constexpr (CLU) {
            ptx::mbar_init(peers_free, uint32_t(p.red_cluster - 1));
            ptx::mbar_init(recv_full, 1);
            *clu_bad = 0u;
        }
        ptx::fence_mbar_init();
        if constexpr (CLU) {
            // The phase completes once the other CTAs' rows (one slot each)
            // have landed.
            ptx::mbar_arrive_expect_tx(recv_full, uint32_t(p.red_cluster - 1) *
                                                      uint32_t(Cfg::ROWS / p.red_cluster) * BN * 4u);
        }
        ptx::prefetch_tensormap(&map_a);
        ptx::prefetch_tensormap(&map_b);
        ptx::prefetch_tensormap(&map_out);
        if (p.fused) {
            ptx::prefetch_tensormap(&map_ws);
            ptx::prefetch_tensormap(&map_red);
        }
    }
    __syncwarp();
    if constexpr (CLU)
        ptx::cluster_arrive_relaxed();  // barriers published; waited on before the first remote access
    if constexpr (PAIR)
        ptx::cluster_sync();  // the peer's barriers exist before anything signals them
    if (warp == 1) {
        ptx::tmem_alloc<PAIR>(ptx::smem_addr(tmem_slot), Cfg::TMEM_COLS);
        ptx::tmem_relinquish<PAIR>();
    } else if (warp == 2 && p.group_rows) {
        build_group_table(p.group_rows, p.groups, p.M, Cfg::TILE_M, p.tiles_n, gtab, p.status);
    }
    ptx::tc_fence_before_sync();
    ptx::cta_sync();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Work units of this launch: fixed, or (grouped) the tiles of all groups.
    const int64_t num_units = p.group_rows ? int64_t(gtab[p.groups - 1]) : p.num_units;
    if (threadIdx.x == 0)
        trace_stamp(p, kTraceSetup);

    AbortFlags af;
    af.local = abort_flag;
    af.peer = PAIR ? ptx::mapa_shared(ptx::smem_addr(const_cast<uint32_t *>(abort_flag)), rank ^ 1u)
                   : 0u;
    af.timeout_ns = p.timeout_ns;
    af.status = p.status;
    // The leader's `full` and `tempty` barriers as shared::cluster addresses.
    const uint32_t full_lead0 = PAIR ? ptx::mapa_shared(full0, 0) : full0;
    const uint32_t tempty_lead0 = PAIR ? ptx::mapa_shared(tempty0, 0) : tempty0;
    const int32_t row_off = PAIR ? int32_t(rank) * kTileM : 0;  // this CTA's rows

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (each CTA fills its own ring)
            uint32_t stage = 0, phase = 0;
            uint64_t issued = 0;
            bool ok = true;
            for (int64_t u = cluster; ok && u < num_units; u += nclusters) {
                const Unit w = decode_unit(u, p, gtab, Cfg::TILE_M, BN);
                // This CTA's B columns: half of each MMA's in a pair, in
                // boxes of 64 columns; box j at bcol(j).
                const int nbox = w.width / (PAIR ? 128 : 64);
                const int32_t col_off = PAIR ? int32_t(rank) * (min(w.width, Cfg::MMA_N) / 2) : 0;
                auto bcol = [&](int j) {
                    return w.n0 + col_off + (j / Cfg::B_BOXES_PER_MMA) * Cfg::MMA_N +
                           64 * (j % Cfg::B_BOXES_PER_MMA);
                };
                const uint32_t tx = uint32_t(Cfg::A_BYTES + nbox * Cfg::B_BOX_BYTES);
                if (p.prefetch_l2) {
                    // The unit's whole K range of A and B at once: DRAM sees the
                    // requests together (better page locality than the ring's
                    // few k-blocks in flight); the ring's loads then hit L2.
                    for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                        ptx::tma_prefetch_l2_3d(&map_a, kb * kTileK, w.m0 + row_off, w.z_in);
#pragma unroll
                        for (int j = 0; j < Cfg::B_BOXES; ++j)
                            if (j < nbox)
                                ptx::tma_prefetch_l2_3d(&map_b, bcol(j), kb * kTileK, w.z_in);
                    }
                }
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, af, kStatusProducer, true)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * Cfg::STAGE_BYTES;
                    if constexpr (PAIR) {
                        // Both CTAs' bytes are counted on the leader's barrier.
                        const uint32_t fb = full_lead0 + 8u * stage;
                        if (leader)
                            ptx::mbar_arrive_expect_tx(full0 + 8u * stage, 2u * tx);
                        ptx::tma_load_3d_pair(sa, &map_a, fb, kb * kTileK, w.m0 + row_off, w.z_in);
#pragma unroll
                        for (int j = 0; j < Cfg::B_BOXES; ++j)
                            if (j < nbox)
                                ptx::tma_load_3d_pair(sa + Cfg::A_BYTES + j * Cfg::B_BOX_BYTES, &map_b,
                                                      fb, bcol(j), kb * kTileK, w.z_in);
                    } else {
                        const uint32_t fb = full0 + 8u * stage;
                        ptx::mbar_arrive_expect_tx(fb, tx);
                        ptx::tma_load_3d(sa, &map_a, fb, kb * kTileK, w.m0, w.z_in);
#pragma unroll
                        for (int j = 0; j < Cfg::B_BOXES; ++j)
                            if (j < nbox)
                                ptx::tma_load_3d(sa + Cfg::A_BYTES + j * Cfg::B_BOX_BYTES, &map_b, fb,
                                                 w.n0 + 64 * j, kb * kTileK, w.z_in);
                    }
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (leader) {
                // Wait (bounded) for the last loads to land, so that no TMA
                // write into shared memory outlives the CTA.  In a pair the
                // leader's barrier also counts the peer's bytes.
                const uint64_t last = issued < uint64_t(S) ? issued : uint64_t(S);
                for (uint64_t i = 0; i < last; ++i) {
                    const uint64_t t = issued - 1 - i;
                    wait_bounded(full0 + 8u * uint32_t(t % S), uint32_t((t / S) & 1u), af,
                                 kStatusDrain, false);
                }
            } else if (*abort_flag) {
                // The peer has no barrier of its own for its loads: after an
                // abort give them a fixed grace period to land.
                const uint64_t t0 = ptx::globaltimer_ns();
                while (ptx::globaltimer_ns() - t0 < 200000ull) {
                }
            }
        }
        __syncwarp();  // lanes 1..31 wait for lane 0 before the CTA barrier
        if constexpr (CLU)
            ptx::cluster_wait();  // the setup arrive's phase, before the exit's
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (one thread; the leader of a pair)
            // Instruction descriptors of a whole tile and of the column
            // slices a narrow tail cuts it into (halves and quarters).
            constexpr uint32_t idesc = mma_idesc<Cfg::MMA_N, PAIR>();
            constexpr uint32_t idesc2 = mma_idesc<Cfg::MMA_N / 2, PAIR>();
            constexpr uint32_t idesc4 = mma_idesc<Cfg::MMA_N / 4, PAIR>();
            constexpr uint16_t both = PAIR ? 3 : 1;
            uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
            bool ok = true;
            for (int64_t u = cluster; ok && u < num_units; u += nclusters) {
                const Unit w = decode_unit(u, p, gtab, Cfg::TILE_M, BN);
                if (!wait_bounded(tempty0 + 8u * abuf, aphase ^ 1u, af, kStatusMma, true)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d = tmem_base + abuf * uint32_t(BN);
                const uint32_t id = w.width == BN ? idesc : (w.width == BN / 2 ? idesc2 : idesc4);
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_bounded(full0 + 8u * stage, phase, af, kStatusMma, true)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    if (u == cluster && kb == w.kb0)
                        trace_stamp(p, kTraceFirstData);
                    const uint32_t sa = base + stage * Cfg::STAGE_BYTES;
                    const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kTileK / 16; ++kk) {
                        // A: advance 16 f16 = 32 bytes along the swizzled row.
                        // B: advance 16 K rows = 2048 bytes.  A 512-column tile:
                        // the second half's B boxes follow the first's.
#pragma unroll
                        for (int hh = 0; hh < Cfg::MMA_HALVES; ++hh)
                            ptx::mma_f16_ss<PAIR>(
                                d + uint32_t(hh * Cfg::MMA_N),
                                desc_a(sa + 32u * kk),
                                desc_b(sb + uint32_t(hh * Cfg::B_BOXES_PER_MMA * Cfg::B_BOX_BYTES) + 2048u * kk),
                                id, (kb > w.kb0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit<PAIR>(empty0 + 8u * stage, both);  // slot free in both CTAs
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                ptx::mma_commit<PAIR>(tfull0 + 8u * abuf, both);  // accumulator ready
                if (++abuf == uint32_t(Cfg::ACC)) {
                    abuf = 0;
                    aphase ^= 1u;
                }
            }
            trace_stamp(p, kTraceLastMma);
            // Every MMA this thread issued must finish before TMEM is freed.
            ptx::mma_commit<PAIR>(done_bar, 1);
            wait_bounded(done_bar, 0, af, kStatusDrain, false);
        }
        __syncwarp();  // lanes 1..31 wait for lane 0 before the CTA barrier
        if constexpr (CLU)
            ptx::cluster_wait();  // the setup arrive's phase, before the exit's
    } else if constexpr (CLU) {
        // ---------------- epilogue of a cluster split-K sum: warps 2..5
        cluster_sum_epilogue<BN, EPI>(p, map_ws, map_red, base, base_ptr, tmem_base, tfull0, stall_bar,
                                      red_bar, peers_free, recv_full, red_ok, clu_bad, abort_flag, af,
                                      num_units, warp, lane);
    } else {
        // ---------------- epilogue: warps 2..5, TMEM lane quarter = warp % 4
        const int e = warp - 2;
        const int q = warp & 3;
        const int h = e >> 2;  // which of the quarter's warps (0 unless HW == 2)
        const uint32_t bufs = epi0 + uint32_t(e) * uint32_t(NBUF) * Cfg::EPI_BUF_BYTES;
        uint32_t abuf = 0, aphase = 0, sbuf = 0;
        if (p.fused && blockIdx.x == 0 && threadIdx.x == 64)
            publish_counters(p.counters, p.counter_words, p.epoch_tag, p.epoch);
        // Split units first (CTA pairs): as soon as the cluster's split unit
        // has stored its partial, its epilogue warps take their share of the
        // tile's sum -- arrive on the tile's counter, wait (bounded) for the
        // tile's split_k x 2 reducers, read rows_per rows of every split from
        // the workspace through L2 and add them in ascending split order into
        // C -- while the MMA warp already works on the cluster's next tile in
        // the other accumulator.  All four epilogue warps pass the three named
        // barriers on every path.
        auto split_sum_from_l2 = [&](const Unit &w) {
            if (lane == 0) {
                ptx::bulk_wait_group_all();  // this warp's partial boxes are written
                ptx::fence_proxy_async_global();
            }
            const int et = int(threadIdx.x) - 64;
            uint64_t epoch_now = 0;
            if (et == 0)
                epoch_now = ptx::ld_relaxed_gpu(p.epoch_tag);
            ptx::named_bar_sync(1, ET);
            const int32_t r0 = (w.s * 2 + int32_t(rank)) * p.rows_per;
            const bool active = r0 < Cfg::TILE_M && w.m0 + r0 < p.M;
            if (et == 0) {
                uint32_t okv = 0;
                const bool epoch_ok = epoch_now == p.epoch ||
                    poll_bounded<unsigned long long>(p.epoch_tag, p.epoch, af, kStatusReduce);
                if (!*abort_flag && epoch_ok) {
                    uint32_t *count = p.counters + w.red_tile;
                    __threadfence();
                    atomicAdd(count, 1u);  // arrive
                    okv = poll_bounded<uint32_t>(count, uint32_t(p.reducers), af, kStatusReduce);
                }
                *red_ok = okv;
            }
            ptx::named_bar_sync(1, ET);  // the acquire above orders the reads below
            if (*red_ok && active) {
                constexpr int U = 4;                                  // chunks in flight per thread
                const int32_t per_row = BN / 4;                       // float4s of a row
                // Only rows inside the tile are read: the last reducer's
                // share may be short, and past the last partial the
                // workspace ends (0 <= r0 < tile_m here).
                const int32_t nf = min(p.rows_per, Cfg::TILE_M - r0) * per_row;
                const int64_t part = int64_t(Cfg::TILE_M) * per_row;  // float4s of one partial
                const float4 *src = reinterpret_cast<const float4 *>(p.ws) +
                                    int64_t(w.red_tile) * p.split_k * part + int64_t(r0) * per_row;
                const float *bias = EPI && p.epi.bias ? p.epi.bias + int64_t(w.z_in) * p.epi.bias_stride : nullptr;
                auto run = [&](auto act) {
                    for (int32_t f0 = et; f0 < nf; f0 += ET * U) {
                        float4 a[U];
#pragma unroll
                        for (int k = 0; k < U; ++k)
                            a[k] = f0 + ET * k < nf ? __ldcg(src + f0 + ET * k) : make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int32_t s2 = 1; s2 < p.split_k; ++s2) {
                            float4 v[U];
#pragma unroll
                            for (int k = 0; k < U; ++k)
                                v[k] = f0 + ET * k < nf ? __ldcg(src + s2 * part + f0 + ET * k) : a[k];
#pragma unroll
                            for (int k = 0; k < U; ++k) {
                                a[k].x += v[k].x;
                                a[k].y += v[k].y;
                                a[k].z += v[k].z;
                                a[k].w += v[k].w;
                            }
                        }
#pragma unroll
                        for (int k = 0; k < U; ++k) {
                            const int32_t f = f0 + ET * k;
                            const int32_t row = f / per_row;
                            const int32_t gr = w.m0 + r0 + row;
                            const int32_t gc = w.n0 + (f - row * per_row) * 4;
                            if (f >= nf || r0 + row >= Cfg::TILE_M || gr >= p.M || gc >= p.N)
                                continue;
                            const int64_t at = int64_t(w.z_in) * p.stride_c + int64_t(gr) * p.ldc + gc;
                            float4 v = a[k];
                            if constexpr (EPI)
                                epi_apply4_as<decltype(act)::value>(v, gc, p.N, bias, p.epi);
                            if (gc + 3 < p.N && (!EPI || p.epi.out_type == kOutF32)) {
                                *reinterpret_cast<float4 *>(static_cast<float *>(p.c_direct) + at) = v;
                            } else if (EPI && gc + 3 < p.N) {
                                *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.c_direct) + at) =
                                    make_uint2(epi_out16(v.x, p.epi.out_type) | (epi_out16(v.y, p.epi.out_type) << 16),
                                               epi_out16(v.z, p.epi.out_type) | (epi_out16(v.w, p.epi.out_type) << 16));
                            } else {
                                const float vv[3] = {v.x, v.y, v.z};
#pragma unroll
                                for (int t = 0; t < 3; ++t)
                                    if (gc + t < p.N)
                                        epi_store(p.c_direct, at + t, vv[t], EPI ? p.epi.out_type : kOutF32);
                            }
                        }
                    }
                };
                if constexpr (EPI)
                    with_activation<ACT>(p.epi.act, run);
                else
                    run(ActTag<kActNone>{});
            }
            ptx::named_bar_sync(1, ET);
            if (et == 0)
                trace_stamp(p, kTraceReduced);
        };
        for (int64_t u = cluster; u < num_units; u += nclusters) {
            const Unit w = decode_unit(u, p, gtab, Cfg::TILE_M, BN);
            bool got = wait_bounded(tfull0 + 8u * abuf, aphase, af, kStatusEpilogue, true);
            if (p.inject_stall && got)
                got = wait_bounded(stall_bar, 0, af, kStatusEpilogue, true);
            if (!__all_sync(0xffffffffu, got)) {
                if constexpr (PAIR) {
                    // A wait ran out and raised the abort flag, so every later
                    // wait returns at once.  With split units first the warps
                    // still walk the remaining units, so that all four pass
                    // the same named barriers in each split sum (which, seeing
                    // the flag, neither arrives nor waits).
                    if (p.split_first) {
                        if (w.split)
                            split_sum_from_l2(w);
                        continue;
                    }
                }
                break;
            }
            ptx::tc_fence_after_sync();
            if (warp == 2 && lane == 0)
                trace_stamp(p, kTraceAccReady);
            const int32_t row0 = w.m0 + row_off + 32 * q;
            // A column slice of the last tile column may start at or past N:
            // then nothing is stored, and the accumulator is still released.
            int nch = 0;
            if (row0 < w.rows && w.n0 < p.N) {
                const int live = (p.N - w.n0 + 31) / 32;
                nch = live < w.width / 32 ? live : w.width / 32;
            }
            const uint32_t tm_row = tmem_base + (uint32_t(32 * q) << 16) + abuf * uint32_t(BN);
            const int32_t tail_row = row0 + lane;
            // A grouped launch's C map spans all M rows, so a warp whose rows
            // cross the group's count writes its rows below it with plain
            // stores instead of TMA.
            const bool rows_partial = p.group_rows != nullptr && row0 + 32 > w.rows;
            // Row `lane` of a 32 x 32 box into `buf`, 16-byte chunk j at
            // (j ^ row % 8): the layout the tensor maps' 128-byte swizzle expects.
            auto stage_box = [&](uint32_t buf, const uint32_t (&r)[32]) {
                const uint32_t row_addr = buf + uint32_t(lane) * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    ptx::st_shared_v4(row_addr + (uint32_t(j ^ (lane & 7)) << 4), r[4 * j],
                                      r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            };
            // Box c goes out by TMA: a split partial to the compact workspace,
            // or the columns of C below n_tma (whole 32-row boxes only).
            auto via_tma = [&](int c) { return w.split || (!rows_partial && w.n0 + 32 * c < p.n_tma); };
            auto store_box = [&](int c, uint32_t buf) {  // lane 0
                if (w.split)
                    ptx::tma_store_3d(&map_ws, buf, 32 * c, row_off + 32 * q, w.z_out);
                else
                    ptx::tma_store_3d(&map_out, buf, w.n0 + 32 * c, row0, w.z_out);
            };
            // Plain stores: columns [n_tma, N) of C (fewer than one 16-byte
            // granule), or the whole row of a warp that crosses its group's
            // row count.
            auto tail_box = [&](int c, const uint32_t (&r)[32]) {
                const int32_t col0 = w.n0 + 32 * c;
                const int32_t from = rows_partial ? col0 : p.n_tma;
                if (!w.split && (rows_partial || (p.tail && col0 + 32 > p.n_tma)) && tail_row < w.rows) {
                    const int64_t row_at = int64_t(w.z_out) * p.stride_c + int64_t(tail_row) * p.ldc;
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int32_t col = col0 + t;
                        if (col >= from && col < p.N)
                            static_cast<float *>(p.c_direct)[row_at + col] = __uint_as_float(r[t]);
                    }
                }
            };
            // Fused epilogue of one box on registers: row `lane`'s 32 values
            // as they come from TMEM, act(alpha * v + bias) with the
            // activation a compile-time constant, so that the 32 values'
            // dependent chains overlap; then staged once for the TMA store --
            // f32 rows in the 128-byte swizzle, or 16-bit rows of 64 bytes in
            // the 64-byte swizzle (16-byte chunk k of row r at k ^ (r / 2) % 4).
            // The bias columns are read as four-float vectors when they are
            // aligned and all inside N (every lane the same address).
            auto reg_box = [&](auto act, uint32_t buf, int c, const uint32_t (&r)[32]) {
                constexpr int A = decltype(act)::value;
                const int32_t col0 = w.n0 + 32 * c;
                const float *bias =
                    p.epi.bias ? p.epi.bias + int64_t(w.z_out) * p.epi.bias_stride + col0 : nullptr;
                float b[32];
                if (bias && col0 + 32 <= p.N && (reinterpret_cast<uintptr_t>(bias) & 15u) == 0) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 t = __ldg(reinterpret_cast<const float4 *>(bias) + j);
                        b[4 * j] = t.x;
                        b[4 * j + 1] = t.y;
                        b[4 * j + 2] = t.z;
                        b[4 * j + 3] = t.w;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        b[k] = bias && col0 + k < p.N ? __ldg(bias + k) : 0.f;
                }
                float v[32];
                const float al = p.epi.alpha, sl = p.epi.slope;
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    v[k] = epi_act(fmaf(al, __uint_as_float(r[k]), b[k]), A, sl);
                if (p.epi.out_type == kOutF32) {
                    const uint32_t row_addr = buf + uint32_t(lane) * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        ptx::st_shared_v4(row_addr + (uint32_t(j ^ (lane & 7)) << 4), __float_as_uint(v[4 * j]),
                                          __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                                          __float_as_uint(v[4 * j + 3]));
                } else {
                    const uint32_t row16 = buf + uint32_t(lane) * 64u;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t hw[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            hw[i] = epi_out16(v[8 * k + 2 * i], p.epi.out_type) |
                                    (epi_out16(v[8 * k + 2 * i + 1], p.epi.out_type) << 16);
                        ptx::st_shared_v4(row16 + (uint32_t(k ^ ((lane >> 1) & 3)) << 4), hw[0], hw[1], hw[2], hw[3]);
                    }
                }
            };
            // Plain stores of an epilogue box from shared memory: the columns
            // the TMA store does not cover, or the rows below a group's count.
            auto epi_tail = [&](uint32_t buf, int c) {
                const int32_t col0 = w.n0 + 32 * c;
                const int32_t from = rows_partial ? col0 : p.n_tma;
                if (!(rows_partial || (p.tail && col0 + 32 > p.n_tma)) || tail_row >= w.rows)
                    return;
                const int64_t row_at = int64_t(w.z_out) * p.stride_c + int64_t(tail_row) * p.ldc;
                const int32_t t0 = max(from - col0, 0);
                const int32_t t1 = min(p.N - col0, 32);
#pragma unroll 1
                for (int32_t t = t0; t < t1; ++t) {
                    if (p.epi.out_type == kOutF32)
                        static_cast<uint32_t *>(p.c_direct)[row_at + col0 + t] = ptx::ld_shared_u32(
                            buf + uint32_t(lane) * 128u + (uint32_t((t >> 2) ^ (lane & 7)) << 4) + uint32_t(t & 3) * 4u);
                    else
                        static_cast<uint16_t *>(p.c_direct)[row_at + col0 + t] = ptx::ld_shared_u16(
                            buf + uint32_t(lane) * 64u + (uint32_t((t >> 3) ^ ((lane >> 1) & 3)) << 4) + uint32_t(t & 7) * 2u);
                }
            };
            // Last read of this accumulator: hand it back to the MMA issuer.
            auto release_acc = [&]() {
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        ptx::mbar_arrive_cluster(tempty_lead0 + 8u * abuf);
                    else
                        ptx::mbar_arrive(tempty0 + 8u * abuf);
                }
            };
            // On the CTA's last unit the operand ring is idle: each box gets
            // a buffer of its own there and no store waits for another.
            const bool drain = Cfg::DRAIN_FITS && u + nclusters >= num_units;
            auto take_buf = [&](int c) -> uint32_t {
                if (drain)
                    return base + (uint32_t(e) * uint32_t(BN / 32 / HW) + uint32_t(c / HW)) * Cfg::EPI_BUF_BYTES;
                if constexpr (NBUF == 2) {
                    if (lane == 0)
                        ptx::bulk_wait_group_read<1>();  // the store that used this buffer has read it
                    __syncwarp();
                    const uint32_t b = bufs + sbuf * Cfg::EPI_BUF_BYTES;
                    sbuf ^= 1u;
                    return b;
                } else {
                    if (lane == 0)
                        ptx::bulk_wait_group_read<0>();  // the warp's previous store has read it
                    __syncwarp();
                    return bufs;
                }
            };
            // One box of the plain epilogue: staged and stored by TMA, and
            // the columns the TMA store does not cover by plain stores.
            auto plain_box = [&](int c, const uint32_t (&r)[32]) {
                if (via_tma(c)) {
                    const uint32_t buf = take_buf(c);
                    stage_box(buf, r);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        store_box(c, buf);
                        ptx::bulk_commit_group();
                    }
                }
                tail_box(c, r);
            };
            // The 512-column tile's accumulator is the only one, and the
            // next tile's MMAs wait until it is read out, which the TMA
            // stores pace (about 43 GB/s per SM): each warp reads its last
            // four boxes into registers at once and hands the accumulator
            // back before it stores them.
            int nloop = nch;
            if constexpr (BN == 512 && !EPI) {
                static_assert(HW == 1, "one epilogue warp per TMEM lane quarter");
                if (!w.split) {
                    constexpr int R = 4;
                    const int nreg = nch < R ? nch : R;
                    for (int c = 0; c < nch - nreg; ++c) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(tm_row + 32u * c, r);
                        ptx::tmem_wait_ld();
                        plain_box(c, r);
                    }
                    if (nreg > 0) {
                        uint32_t rr[R][32];
#pragma unroll
                        for (int i = 0; i < R; ++i)
                            if (i < nreg)
                                ptx::tmem_ld_32x32b_x32(tm_row + 32u * uint32_t(nch - nreg + i), rr[i]);
                        ptx::tmem_wait_ld();
                        release_acc();
#pragma unroll
                        for (int i = 0; i < R; ++i)
                            if (i < nreg)
                                plain_box(nch - nreg + i, rr[i]);
                    }
                    nloop = 0;
                }
            }
            // This warp's boxes: all of them, or every HW-th from h.
            for (int c = h; c < nloop; c += HW) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tm_row + 32u * c, r);
                ptx::tmem_wait_ld();
                if (c + HW >= nch)
                    release_acc();
                const bool tma = via_tma(c);
                if constexpr (EPI) {
                    if (!w.split) {
                        const uint32_t buf = take_buf(c);
                        with_activation<ACT>(p.epi.act, [&](auto act) { reg_box(act, buf, c, r); });
                        if (tma) {
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                store_box(c, buf);
                                ptx::bulk_commit_group();
                            }
                        }
                        epi_tail(buf, c);
                        continue;
                    }
                }
                if (tma) {
                    const uint32_t buf = take_buf(c);
                    stage_box(buf, r);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        store_box(c, buf);
                        ptx::bulk_commit_group();
                    }
                }
                tail_box(c, r);
            }
            if (h >= nch)  // no box for this warp
                release_acc();
            if (++abuf == uint32_t(Cfg::ACC)) {
                abuf = 0;
                aphase ^= 1u;
            }
            if constexpr (PAIR) {
                if (p.split_first && w.split)
                    split_sum_from_l2(w);
            }
        }
        if (lane == 0)
            ptx::bulk_wait_group_all();  // stores complete before the CTA exits
        __syncwarp();
        if (warp == 2 && lane == 0)
            trace_stamp(p, kTraceStored);

        // The CTA's last assigned unit decides whether it takes part in an
        // in-kernel split-K sum (computed from the assignment, not from how
        // far the loop got, so all four warps agree even after an abort).
        int64_t last_u = -1;
        if (cluster < num_units)
            last_u = cluster + (num_units - 1 - cluster) / nclusters * nclusters;
        const Unit w = last_u >= 0 ? decode_unit(last_u, p, gtab, Cfg::TILE_M, BN) : Unit{};
        if (p.fused && !p.split_first && last_u >= 0 && w.split) {
            // ---------------- in-kernel split-K sum
            // The CTA's partial is in the workspace (its TMA stores completed
            // above); the CTA arrives on its tile's counter, waits (bounded)
            // until all reducers = split_k x CTAs-per-unit have arrived, fetches
            // rows_per rows of every split of the tile with one TMA load into
            // the idle ring, sums them in ascending split order (the order of
            // the separate reduce kernel, so the sums are bitwise the same) and
            // writes C.  All four epilogue warps pass the three named barriers
            // on every path.
            const int et = int(threadIdx.x) - 64;  // 0 .. ET - 1
            // The counters belong to this launch once CTA 0 has published the
            // epoch, normally long before now: read it early (relaxed) and
            // check it after the barrier; the GPU-scope fence before the
            // arrival completes the acquire.
            uint64_t epoch_now = 0;
            if (et == 0)
                epoch_now = ptx::ld_relaxed_gpu(p.epoch_tag);
            // Each warp's TMA stores are complete (waited above); the proxy
            // fence orders them before the warp's later generic accesses, the
            // barrier before the arriving thread's, and that thread's
            // GPU-scope fence (cumulative) before its arrival.
            if (lane == 0)
                ptx::fence_proxy_async_global();
            ptx::named_bar_sync(1, ET);
            const int64_t bz = w.z_in;
            const int32_t ri = w.s * (PAIR ? 2 : 1) + int32_t(rank);
            const int32_t r0 = ri * p.rows_per;               // first tile row this CTA sums
            const bool active = r0 < Cfg::TILE_M && w.m0 + r0 < p.M;
            const uint32_t box_bytes = uint32_t(p.rows_per) * BN * 4u * uint32_t(p.split_k);
            if (et == 0) {
                uint32_t okv = 0;
                const bool epoch_ok = epoch_now == p.epoch ||
                    poll_bounded<unsigned long long>(p.epoch_tag, p.epoch, af, kStatusReduce);
                if (!*abort_flag && epoch_ok) {
                    uint32_t *count = p.counters + w.red_tile;
                    __threadfence();
                    atomicAdd(count, 1u);  // arrive
                    okv = poll_bounded<uint32_t>(count, uint32_t(p.reducers), af, kStatusReduce);
                    if (okv && active) {
                        // The acquire that saw the count orders this load
                        // after every split's partial.
                        ptx::fence_proxy_async_global();
                        ptx::mbar_arrive_expect_tx(red_bar, box_bytes);
                        // box {BN columns, rows_per rows, split_k splits} of the
                        // compact workspace, starting at this tile's first split
                        ptx::tma_load_3d(base, &map_red, red_bar, 0, r0,
                                         int32_t(w.red_tile * p.split_k));
                    }
                }
                *red_ok = okv;
            }
            ptx::named_bar_sync(1, ET);
            if (*red_ok && active) {
                // The load is in flight and finishes on its own: wait it out.
                if (wait_bounded(red_bar, 0, af, kStatusReduce, false)) {
                    const float4 *stg = reinterpret_cast<const float4 *>(base_ptr);
                    const int32_t per_split = p.rows_per * (BN / 4);  // float4s of one split
                    const int32_t nsplit = p.split_k;
                    auto put = [&](auto act, int32_t f, const float4 &acc) {
                        const int32_t row = f / (BN / 4);
                        const int32_t gr = w.m0 + r0 + row;
                        const int32_t gc = w.n0 + (f - row * (BN / 4)) * 4;
                        if (row < p.rows_per && r0 + row < Cfg::TILE_M && gr < p.M && gc < p.N) {
                            const int64_t at = bz * p.stride_c + int64_t(gr) * p.ldc + gc;
                            if constexpr (EPI) {
                                const float *bias =
                                    p.epi.bias ? p.epi.bias + bz * p.epi.bias_stride : nullptr;
                                float4 v = acc;
                                epi_apply4_as<decltype(act)::value>(v, gc, p.N, bias, p.epi);
                                if (gc + 3 < p.N && p.epi.out_type == kOutF32) {
                                    *reinterpret_cast<float4 *>(static_cast<float *>(p.c_direct) + at) = v;
                                } else if (gc + 3 < p.N) {
                                    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.c_direct) + at) =
                                        make_uint2(epi_out16(v.x, p.epi.out_type) |
                                                       (epi_out16(v.y, p.epi.out_type) << 16),
                                                   epi_out16(v.z, p.epi.out_type) |
                                                       (epi_out16(v.w, p.epi.out_type) << 16));
                                } else {
                                    const float vv[3] = {v.x, v.y, v.z};
#pragma unroll
                                    for (int k = 0; k < 3; ++k)
                                        if (gc + k < p.N)
                                            epi_store(p.c_direct, at + k, vv[k], p.epi.out_type);
                                }
                            } else {
                                float *dst = static_cast<float *>(p.c_direct) + at;
                                if (gc + 3 < p.N) {
                                    *reinterpret_cast<float4 *>(dst) = acc;
                                } else {
                                    dst[0] = acc.x;
                                    if (gc + 1 < p.N)
                                        dst[1] = acc.y;
                                    if (gc + 2 < p.N)
                                        dst[2] = acc.z;
                                }
                            }
                        }
                    };
                    // Two float4s per thread per pass, splits unrolled: the
                    // shared-memory loads overlap, while each sum still adds
                    // the splits one at a time in ascending order.  The
                    // activation is a compile-time constant of the loop (one
                    // dispatch per CTA), so the values' activations overlap.
                    auto sum_all = [&](auto act) {
                        for (int32_t f0 = et; f0 < per_split; f0 += 2 * ET) {
                            const int32_t f1 = f0 + ET;
                            const bool two = f1 < per_split;
                            float4 a0 = stg[f0];
                            float4 a1 = two ? stg[f1] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
                            for (int32_t s2 = 1; s2 < nsplit; ++s2) {
                                const float4 v0 = stg[s2 * per_split + f0];
                                const float4 v1 = two ? stg[s2 * per_split + f1] : v0;
                                a0.x += v0.x;
                                a0.y += v0.y;
                                a0.z += v0.z;
                                a0.w += v0.w;
                                a1.x += v1.x;
                                a1.y += v1.y;
                                a1.z += v1.z;
                                a1.w += v1.w;
                            }
                            put(act, f0, a0);
                            if (two)
                                put(act, f1, a1);
                        }
                    };
                    if constexpr (EPI)
                        with_activation<ACT>(p.epi.act, sum_all);
                    else
                        sum_all(ActTag<kActNone>{});
                }
            }
            ptx::named_bar_sync(1, ET);
            if (et == 0)
                trace_stamp(p, kTraceReduced);
        }
    }

    ptx::tc_fence_before_sync();
    ptx::cta_sync();
    if constexpr (PAIR || CLU)
        ptx::cluster_sync();  // no CTA leaves while another of its cluster may still signal it
    if (threadIdx.x == 64)    // an epilogue thread: the last role to finish
        trace_stamp(p, kTraceExit);
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc<PAIR>(tmem_base, Cfg::TMEM_COLS);
    }
}

// ------------------------------------------------------------- launching

template <int BN, bool PAIR, bool EPI, bool CLU, int ACT>
inline cudaError_t set_attr()
{
    return cudaFuncSetAttribute(tsm_gemm_tcgen05_kernel<BN, PAIR, EPI, CLU, ACT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TileCfg<BN, PAIR>::SMEM_BYTES);
}

template <int BN, bool PAIR, bool EPI, bool CLU, int ACT>
inline cudaError_t launch_bn(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                             const CUtensorMap &ws, const CUtensorMap &r, const KernelParams &p,
                             int grid, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(gemm_threads(EPI, CLU), 1, 1);
    cfg.dynamicSmemBytes = TileCfg<BN, PAIR>::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (PAIR || CLU) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = PAIR ? 2u : unsigned(p.red_cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    } else {
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
    }
    return cudaLaunchKernelEx(&cfg, tsm_gemm_tcgen05_kernel<BN, PAIR, EPI, CLU, ACT>, a, b, o, ws, r, p);
}

}  // namespace tsm
