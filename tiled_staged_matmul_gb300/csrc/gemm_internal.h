// gemm_internal.h -- what the host planner (gemm_api.cu) and the kernel
// translation unit (gemm_kernels.cu) share.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace tsm {

constexpr int kTileM = 128;  // rows of C per tile = TMEM lanes of one accumulator
constexpr int kTileK = 64;   // K depth of one k-block: one 128-byte swizzle row of f16
constexpr int kThreads = 192;  // warp 0 TMA producer, warp 1 MMA issuer, warps 2..5 epilogue

// Epilogue warps of a GEMM kernel: two per TMEM lane quarter with a fused
// epilogue (not in the cluster split-K sum), else one.
__host__ __device__ constexpr int epilogue_warps(bool epi, bool clu) { return epi && !clu ? 8 : 4; }
// Threads of a GEMM kernel: the producer and MMA warps, then the epilogue's.
__host__ __device__ constexpr int gemm_threads(bool epi, bool clu) { return 64 + 32 * epilogue_warps(epi, clu); }

// Fused epilogue: what the kernels do to an output value before storing it,
// C = act(alpha * acc + bias[j]), stored as `out_type`.  The identity (alpha
// 1, no bias, no activation, f32) is the plain GEMM.
enum : int32_t { kActNone = 0, kActRelu = 1, kActLeakyRelu = 2, kActGelu = 3, kActGeluTanh = 4,
                 kActSilu = 5 };
enum : int32_t { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };
struct Epilogue {
    float alpha = 1.0f;
    const float *bias = nullptr;  // N values per batch, bias_stride apart (0: one for all)
    int64_t bias_stride = 0;
    int32_t act = kActNone;
    float slope = 0.0f;           // kActLeakyRelu
    int32_t out_type = kOutF32;
    __host__ __device__ bool identity() const
    {
        return alpha == 1.0f && !bias && act == kActNone && out_type == kOutF32;
    }
    __host__ __device__ int out_bytes() const { return out_type == kOutF32 ? 4 : 2; }
};

// Bits of the device status word: which role's bounded wait ran out.
constexpr uint32_t kStatusProducer = 1u;
constexpr uint32_t kStatusMma = 2u;
constexpr uint32_t kStatusEpilogue = 4u;
constexpr uint32_t kStatusDrain = 8u;
constexpr uint32_t kStatusReduce = 16u;
constexpr uint32_t kStatusGroupRows = 32u;  // a group's row count outside [0, M] (clamped)

// Grouped launches: at most this many groups per launch (the per-CTA table of
// tile offsets lives in the shared-memory control block).
constexpr int kMaxGroupsPerLaunch = 256;

// Everything the persistent kernel needs besides its three tensor maps.
struct KernelParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n;
    int32_t k_blocks;     // ceil(K / kTileK)
    int32_t split_k;      // K ranges per tile (1 = the output map is C itself)
    int32_t batch;
    int32_t group_m;      // raster: tiles of M walked together
    int32_t inject_stall; // test hook: the epilogue waits on a barrier nothing signals
    int64_t num_units;    // batch * split_k * tiles_m * tiles_n
    uint64_t timeout_ns;  // limit of every device-side wait
    uint32_t *status;     // device status word (OR of kStatus* bits)
    // A TMA store writes whole 16-byte granules of a row, so it covers only
    // the columns below n_tma (a multiple of 4); when `tail` is set the
    // epilogue writes columns [n_tma, N) of C with plain stores.
    int32_t n_tma;
    int32_t tail;
    void *c_direct;       // C itself (tail stores, in-kernel split-K sums), epi.out_type elements
    int64_t ldc;
    int64_t stride_c;
    // In-kernel split-K reduction (each cluster owns exactly one unit): the
    // partials are TMA-stored like those of the separate reduction
    // ([batch * split][M][ldw] f32, through the output map); the
    // split_k x (CTAs per unit) reducers of a tile each own rows_per rows of
    // it, fetch those rows of every split with one TMA load (the reduce map)
    // and sum them in ascending split order.  counters holds one arrival
    // count per split tile (counter_words of them); the workspace holds
    // whatever its last user left there, so CTA 0 zeroes the counters at the
    // start of the launch and then publishes `epoch` (unique to this launch)
    // in *epoch_tag, and a CTA arrives only after it has read that epoch.
    int32_t fused;
    int32_t reducers;
    int32_t rows_per;
    // Cluster split-K sum (with `fused`, every unit a split unit): the grid
    // runs in clusters of red_cluster CTAs (2 or 4) holding red_cluster
    // consecutive K ranges of one tile; CTA rank r of a cluster owns tile rows
    // [r * tile_m / red_cluster, (r + 1) * tile_m / red_cluster), receives
    // those rows of the other CTAs' partials through distributed shared
    // memory and adds them in ascending rank.  The tile's red_groups =
    // split_k / red_cluster cluster partials then go through the compact
    // workspace ([tile * red_groups + g][tile_m][tile_n]) and are summed as
    // above in ascending g, rows_per rows per reducer; counters then hold one
    // word per (tile, rank).  With red_groups == 1 the cluster writes C.
    // 1: off.
    int32_t red_cluster;
    int32_t red_groups;
    // With `fused`, units [0, dp_units) are whole tiles written straight to C
    // (the full waves of a "split tail" plan) and units from dp_units on are
    // split units, tile-major: unit dp_units + j computes split j % split_k
    // of tile dp_units + j / split_k, and its partial goes to the compact
    // workspace [j][tile_m][tile_n] (through the workspace map).
    int64_t dp_units;
    // Split units first (CTA pairs, "split tail" plans whose split units all
    // fit the first wave): units [0, n_first) are the split units j = u and
    // the whole tiles follow (unit n_first + t is tile t).  Each split unit is
    // the first unit of its cluster, its partners run at the same time, and
    // its epilogue warps sum the tile from the workspace (`ws`, read through
    // L2) while the MMA warp already works on the cluster's next tile.
    int32_t split_first;
    int64_t n_first;
    const float *ws;
    // Narrow tail (not with `fused`): units [0, dp_units) are whole tiles,
    // and each later tile is cut into `narrow` column slices of
    // tile_n / narrow columns (2 or 4), each a unit of its own over all of K:
    // the last wave keeps more slots busy without any partial sums.  0: none.
    int32_t narrow;
    int32_t prefetch_l2;  // 1: the producer first asks L2 for its unit's whole K range
    uint32_t *counters;
    int32_t counter_words;
    unsigned long long *epoch_tag;
    unsigned long long epoch;  // never 0
    // Grouped (Mixture-of-Experts) launch: group g = batch index g has
    // group_rows[g] valid rows (device memory, clamped to [0, M]); its tiles
    // are ceil(rows / tile) x tiles_n, numbered after those of groups < g, and
    // rows at or past the count are neither stored nor summed.  Null: every
    // batch has M rows.  groups <= kMaxGroupsPerLaunch.
    const int32_t *group_rows;
    int32_t groups;
    // The fused epilogue (identity for the plain GEMM; only the kernels built
    // with it read it).
    Epilogue epi;
    // Optional per-CTA timeline (kTraceSlots globaltimer stamps per CTA), or null.
    unsigned long long *trace;
};

// Trace slots (ns, %globaltimer), one row of kTraceSlots per CTA.
constexpr int kTraceSlots = 8;
enum TraceSlot {
    kTraceEntry = 0,       // kernel entry
    kTraceSetup = 1,       // barriers, TMEM and tensor maps ready
    kTraceFirstData = 2,   // MMA issuer: first k-block landed in shared memory
    kTraceLastMma = 3,     // MMA issuer: last MMA issued
    kTraceAccReady = 4,    // epilogue: last accumulator ready
    kTraceStored = 5,      // epilogue: output (or partial) written
    kTraceReduced = 6,     // epilogue: in-kernel split-K sum written
    kTraceExit = 7         // before TMEM is freed
};

// Shared-memory budget of one CTA for a tile width (host and device agree).
struct SmemBudget {
    int stages;
    int stage_bytes;
    int smem_bytes;
    int tmem_cols;
};
SmemBudget smem_budget(int tile_m, int tile_n);

// Kernel-side entry points (defined in gemm_kernels.cu).
// `epi`: the kernel built with the fused epilogue (any Epilogue), else the
// plain one (identity Epilogue only).
// `red_cluster` > 1: the kernel built for the cluster split-K sum, launched in
// clusters of that many CTAs (one CTA per tile only).
// `act`: with `epi`, the activation the kernel is built for (the cluster
// split-K sums read it at run time and take any).
cudaError_t set_kernel_attributes(int tile_m, int tile_n, bool epi, int red_cluster = 1, int act = kActNone);
// Clusters of `red_cluster` CTAs of the cluster-sum kernel (tile_n columns)
// that fit on the device at once (cudaOccupancyMaxActiveClusters).
cudaError_t cluster_capacity(int tile_n, int red_cluster, int *clusters);
// The fused-epilogue kernels of one CTA or a pair for activation ACT
// (gemm_epi.cu, one unit per activation).
template <int ACT>
cudaError_t set_epi_attributes(int tile_m, int tile_n);
template <int ACT>
cudaError_t launch_epi(int tile_m, int tile_n, const CUtensorMap &map_a, const CUtensorMap &map_b,
                       const CUtensorMap &map_out, const CUtensorMap &map_ws, const CUtensorMap &map_red,
                       const KernelParams &p, int grid, cudaStream_t stream);
// With `epi` and no cluster sum, the kernel of p.epi.act.
cudaError_t launch_tcgen05_gemm(int tile_m, int tile_n, bool epi, int red_cluster,
                                const CUtensorMap &map_a,
                                const CUtensorMap &map_b, const CUtensorMap &map_out,
                                const CUtensorMap &map_ws, const CUtensorMap &map_red,
                                const KernelParams &p, int grid, cudaStream_t stream);
cudaError_t launch_splitk_reduce(const float *W, void *C, int32_t M, int32_t N, int32_t S,
                                 int32_t batch, int64_t ldw, int64_t ldc, int64_t strideC,
                                 const Epilogue &epi, int grid, cudaStream_t stream);
// Repack A or B into a packed layout with 16-byte aligned rows, and copy a
// result out of one (only the rows below each count when group_rows is set).
cudaError_t launch_pack_f16(const uint16_t *src, int64_t s_ld, int64_t s_stride, uint16_t *dst,
                            int64_t d_ld, int64_t d_stride, int32_t rows, int32_t cols,
                            int32_t batch, int sms, cudaStream_t stream);
cudaError_t launch_unpack_f32(const float *src, int64_t s_ld, int64_t s_stride, float *dst,
                              int64_t d_ld, int64_t d_stride, int32_t rows, int32_t cols,
                              int32_t batch, const int32_t *group_rows, int sms,
                              cudaStream_t stream);
cudaError_t launch_unpack_u16(const uint16_t *src, int64_t s_ld, int64_t s_stride, uint16_t *dst,
                              int64_t d_ld, int64_t d_stride, int32_t rows, int32_t cols,
                              int32_t batch, const int32_t *group_rows, int sms,
                              cudaStream_t stream);
// K == 0: every cell is the epilogue of the empty sum, act(bias[j]).
cudaError_t launch_zero_fill(void *C, int32_t M, int32_t N, int32_t batch, int64_t ldc,
                             int64_t strideC, const int32_t *group_rows, const Epilogue &epi,
                             int grid, cudaStream_t stream);
cudaError_t device_status_word(uint32_t **ptr);

// Row reductions (rowsum_kernels.cu): the tiled row sum and the GEMV.
struct RowReduceParams {
    const void *X;        // element type per the launch (f32, f16, bf16; f16 for the GEMV)
    int64_t row_stride;   // elements
    int64_t col_stride;   // elements (1 on the vector path)
    const uint16_t *xv;   // GEMV: x (f16), incx apart; else null
    int64_t incx;
    float *out;           // R results
    float *partial;       // R * segs partial sums when segs > 1
    int64_t R, C;
    int64_t seg;          // columns per item (a multiple of 16 bytes of elements on the vector path)
    int32_t segs;         // items per row
    int32_t tpr;          // lanes per worker: 1, 2, 4, ..., 32
};
cudaError_t launch_row_reduce(const RowReduceParams &p, int elem, bool vec, bool gemv, int grid,
                              cudaStream_t stream);
// Blocks of 256 threads of that row-reduction kernel one SM holds at once.
int row_reduce_blocks_per_sm(int elem, bool vec, bool gemv);
cudaError_t launch_row_partials(const float *partial, float *out, int64_t R, int32_t segs, int grid,
                                cudaStream_t stream);

}  // namespace tsm
