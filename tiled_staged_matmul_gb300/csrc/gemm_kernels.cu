// gemm_kernels.cu -- the sm_103a kernels of the K-tiled, operand-staged GEMM.
//
// The method ("The PTSS Cliff: A Kernel That Won't Build", sections "The
// Idea: Stage in SLM, Tile K" and "The Pass, Step by Step"): instead of
// holding whole operand tiles in registers, stage them in fast on-chip memory
// and walk K in fixed-size chunks, carrying the accumulator across chunks.
// On GB300 that becomes:
//
//   * staging: a ring of STAGES shared-memory slots, each holding one
//     128 x 64 A tile and one 64 x BN B tile, filled by TMA from tensor maps
//     whose extent masks out-of-range elements to zero ("Intel XPU Backend
//     for Triton", section "Use Tensor Descriptors to load tl.dot arguments
//     and save results");
//   * the K_TILE loop: one 64-deep k-block per slot, four 128 x BN x 16
//     tcgen05 MMAs per k-block, all accumulating into one f32 tile held in
//     tensor memory (TMEM) -- the carried accumulator of the pages' loop;
//   * mbarriers hand each slot from the TMA producer to the MMA issuer
//     (full) and back (empty); two TMEM accumulators let the epilogue drain
//     one tile while the next one accumulates;
//   * the epilogue reads TMEM into registers, writes a swizzled 32 x 32 f32
//     box to shared memory and stores it with TMA, clipped at M and N
//     (the pages' descriptor store, same section);
//   * split-K: a tile's K range may be cut into S contiguous pieces whose
//     f32 partials go to a workspace; a second kernel sums them in ascending
//     split order, so the result never depends on which CTA finished first
//     ("A Dumb Triton Runtime Error", sections "What I ran" and "The Takeaway
//     and the Final Fix": inter-CTA atomics need a zeroed output and change
//     the rounding with the order).
//
// Every mbarrier wait is bounded in time.  A wait that runs out records a
// bit in the device status word and the CTA winds down: it waits (bounded)
// for its own TMA loads, MMAs and stores still in flight, frees its TMEM and
// returns.  Nothing traps.
#include "gemm_kernel.cuh"

namespace tsm {

__device__ uint32_t g_status_word;

// ------------------------------------------------------------- split-K reduce

// C[b][i][j] = sum over s = 0, 1, ..., S-1 (in that order) of
// W[b*S + s][i][j].  Four adjacent columns per thread; W's rows are ldw
// floats (ldw a multiple of 4), so the loads are aligned float4s.
__global__ void __launch_bounds__(256)
    tsm_splitk_reduce_kernel(const float *__restrict__ W, void *__restrict__ C, int32_t M,
                             int32_t N, int32_t S, int32_t batch, int64_t ldw, int64_t ldc,
                             int64_t strideC, Epilogue epi)
{
    const bool plain = epi.identity();
    const int64_t n4 = (N + 3) / 4;
    const int64_t per_mat = int64_t(M) * n4;
    const int64_t total = per_mat * batch;
    const int64_t wmat = int64_t(M) * ldw;
    for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += int64_t(gridDim.x) * blockDim.x) {
        const int64_t b = idx / per_mat;
        const int64_t r = idx - b * per_mat;
        const int64_t i = r / n4;
        const int32_t j = int32_t(r - i * n4) * 4;
        const float *w = W + b * S * wmat + i * ldw + j;
        float4 acc = __ldg(reinterpret_cast<const float4 *>(w));
#pragma unroll 8
        for (int32_t s = 1; s < S; ++s) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(w + int64_t(s) * wmat));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const int64_t at = b * strideC + i * ldc + j;
        if (plain) {
            float *c = static_cast<float *>(C) + at;
            if (j + 3 < N) {
                *reinterpret_cast<float4 *>(c) = acc;
            } else {
                c[0] = acc.x;
                if (j + 1 < N)
                    c[1] = acc.y;
                if (j + 2 < N)
                    c[2] = acc.z;
            }
            continue;
        }
        const float *bias = epi.bias ? epi.bias + b * epi.bias_stride : nullptr;
        const float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (j + k < N)
                epi_store(C, at + k, epi_value(v[k], bias ? __ldg(bias + j + k) : 0.f, epi),
                          epi.out_type);
    }
}

// K == 0: every cell is the empty sum, through the epilogue: act(bias[j])
// (in a grouped launch, every cell of the rows below the group's count,
// clamped to [0, M]).
__global__ void __launch_bounds__(256)
    tsm_zero_fill_kernel(void *__restrict__ C, int32_t M, int32_t N, int32_t batch, int64_t ldc,
                         int64_t strideC, const int32_t *__restrict__ group_rows, Epilogue epi)
{
    const int64_t per_mat = int64_t(M) * N;
    const int64_t total = per_mat * batch;
    for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += int64_t(gridDim.x) * blockDim.x) {
        const int64_t b = idx / per_mat;
        const int64_t r = idx - b * per_mat;
        const int64_t i = r / N;
        const int64_t j = r - i * N;
        if (group_rows && i >= group_rows[b])
            continue;
        const float bv = epi.bias ? __ldg(epi.bias + b * epi.bias_stride + j) : 0.f;
        epi_store(C, b * strideC + i * ldc + j, epi_value(0.f, bv, epi), epi.out_type);
    }
}

// Repacking between a pitched layout the TMA cannot address and a packed
// one whose rows start on 16-byte boundaries: the repack of an operand
// before the GEMM (PACK: the destination is the packed side) and the
// copy-out of a result computed in the packed layout (!PACK: the source is,
// and with `group_rows` only the rows below each batch's count are written).
// Each thread moves 16-byte chunks of a row: one vector access on the
// packed side, element accesses (all of a chunk in flight at once) on the
// other.  Grid: x walks groups of `rows_per_block` rows, y splits a row's
// chunks into segments of `seg` chunks, z walks the batch.
template <typename T, bool PACK>
__global__ void __launch_bounds__(256)
    tsm_repack_kernel(const T *__restrict__ src, int64_t s_ld, int64_t s_stride, T *__restrict__ dst,
                      int64_t d_ld, int64_t d_stride, int32_t rows, int32_t cols, int32_t batch,
                      int32_t tpr, int32_t seg, const int32_t *__restrict__ group_rows)
{
    constexpr int V = 16 / sizeof(T);  // elements per chunk
    const int32_t chunks = (cols + V - 1) / V;
    const int32_t rpb = 256 / tpr;
    const int32_t my_r = int32_t(threadIdx.x) / tpr;
    const int32_t my_c = int32_t(threadIdx.x) - my_r * tpr;
    const int32_t c_begin = int32_t(blockIdx.y) * seg;
    const int32_t c_end = min(chunks, c_begin + seg);
    for (int32_t b = int32_t(blockIdx.z); b < batch; b += int32_t(gridDim.z)) {
        const int32_t lim = group_rows ? min(max(group_rows[b], 0), rows) : rows;
        for (int64_t r = int64_t(blockIdx.x) * rpb + my_r; r < lim; r += int64_t(gridDim.x) * rpb) {
            const T *srow = src + int64_t(b) * s_stride + r * s_ld;
            T *drow = dst + int64_t(b) * d_stride + r * d_ld;
#pragma unroll 2
            for (int32_t c = c_begin + my_c; c < c_end; c += tpr) {
                const int32_t e0 = c * V;
                T v[V];
                if (PACK) {
                    if (e0 + V <= cols) {
#pragma unroll
                        for (int j = 0; j < V; ++j)
                            v[j] = srow[e0 + j];
                    } else {
#pragma unroll
                        for (int j = 0; j < V; ++j)
                            v[j] = e0 + j < cols ? srow[e0 + j] : T(0);
                    }
                    uint4 w;
                    memcpy(&w, v, 16);
                    *reinterpret_cast<uint4 *>(drow + e0) = w;
                } else {
                    const uint4 w = *reinterpret_cast<const uint4 *>(srow + e0);
                    memcpy(v, &w, 16);
                    if (e0 + V <= cols) {
#pragma unroll
                        for (int j = 0; j < V; ++j)
                            drow[e0 + j] = v[j];
                    } else {
#pragma unroll
                        for (int j = 0; j < V; ++j)
                            if (e0 + j < cols)
                                drow[e0 + j] = v[j];
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------- host side

template <int BN, bool PAIR>
static SmemBudget budget_of()
{
    using Cfg = TileCfg<BN, PAIR>;
    return SmemBudget{Cfg::STAGES, Cfg::STAGE_BYTES, Cfg::SMEM_BYTES, int(Cfg::TMEM_COLS)};
}

SmemBudget smem_budget(int tile_m, int tile_n)
{
    if (tile_m == 2 * kTileM)
        return tile_n == 128 ? budget_of<128, true>()
                             : tile_n == 512 ? budget_of<512, true>() : budget_of<256, true>();
    switch (tile_n) {
    case 64: return budget_of<64, false>();
    case 128: return budget_of<128, false>();
    default: return budget_of<256, false>();
    }
}

// The plain kernels (identity epilogue) and the cluster split-K sums (plain,
// or with the epilogue read at run time); the fused-epilogue kernels of one
// CTA or a pair are built per activation in gemm_epi.cu.
static cudaError_t set_plain_or_cluster_attrs(int tile_m, int tile_n, bool epi, int red_cluster)
{
    if (red_cluster > 1) {
        if (tile_m != kTileM)
            return cudaErrorInvalidValue;
        switch (tile_n) {
        case 128: return epi ? set_attr<128, false, true, true, kActRuntime>()
                             : set_attr<128, false, false, true, kActNone>();
        case 256: return epi ? set_attr<256, false, true, true, kActRuntime>()
                             : set_attr<256, false, false, true, kActNone>();
        default: return cudaErrorInvalidValue;
        }
    }
    if (epi)
        return cudaErrorInvalidValue;
    if (tile_m == 2 * kTileM) {
        switch (tile_n) {
        case 128: return set_attr<128, true, false, false, kActNone>();
        case 256: return set_attr<256, true, false, false, kActNone>();
        case 512: return set_attr<512, true, false, false, kActNone>();
        default: return cudaErrorInvalidValue;
        }
    }
    switch (tile_n) {
    case 64: return set_attr<64, false, false, false, kActNone>();
    case 128: return set_attr<128, false, false, false, kActNone>();
    case 256: return set_attr<256, false, false, false, kActNone>();
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t set_kernel_attributes(int tile_m, int tile_n, bool epi, int red_cluster, int act)
{
    if (epi && red_cluster <= 1) {
        switch (act) {
        case kActNone: return set_epi_attributes<kActNone>(tile_m, tile_n);
        case kActRelu: return set_epi_attributes<kActRelu>(tile_m, tile_n);
        case kActLeakyRelu: return set_epi_attributes<kActLeakyRelu>(tile_m, tile_n);
        case kActGelu: return set_epi_attributes<kActGelu>(tile_m, tile_n);
        case kActGeluTanh: return set_epi_attributes<kActGeluTanh>(tile_m, tile_n);
        case kActSilu: return set_epi_attributes<kActSilu>(tile_m, tile_n);
        default: return cudaErrorInvalidValue;
        }
    }
    return set_plain_or_cluster_attrs(tile_m, tile_n, epi, red_cluster);
}

static cudaError_t launch_plain_or_cluster(int tile_m, int tile_n, bool epi, int red_cluster,
                                           const CUtensorMap &map_a, const CUtensorMap &map_b,
                                           const CUtensorMap &map_out, const CUtensorMap &map_ws,
                                           const CUtensorMap &map_red, const KernelParams &p, int grid,
                                           cudaStream_t stream)
{
    if (red_cluster > 1) {
        if (tile_m != kTileM || grid % red_cluster || p.red_cluster != red_cluster)
            return cudaErrorInvalidValue;
        switch (tile_n) {
        case 128:
            return epi ? launch_bn<128, false, true, true, kActRuntime>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream)
                       : launch_bn<128, false, false, true, kActNone>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case 256:
            return epi ? launch_bn<256, false, true, true, kActRuntime>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream)
                       : launch_bn<256, false, false, true, kActNone>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    if (epi)
        return cudaErrorInvalidValue;
    if (tile_m == 2 * kTileM) {
        if (grid % 2)
            return cudaErrorInvalidValue;
        switch (tile_n) {
        case 128: return launch_bn<128, true, false, false, kActNone>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case 256: return launch_bn<256, true, false, false, kActNone>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case 512: return launch_bn<512, true, false, false, kActNone>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (tile_n) {
    case 64: return launch_bn<64, false, false, false, kActNone>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
    case 128: return launch_bn<128, false, false, false, kActNone>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
    case 256: return launch_bn<256, false, false, false, kActNone>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tcgen05_gemm(int tile_m, int tile_n, bool epi, int red_cluster,
                                const CUtensorMap &map_a, const CUtensorMap &map_b,
                                const CUtensorMap &map_out, const CUtensorMap &map_ws,
                                const CUtensorMap &map_red, const KernelParams &p, int grid,
                                cudaStream_t stream)
{
    if (epi && red_cluster <= 1) {
        if (tile_m == 2 * kTileM && grid % 2)
            return cudaErrorInvalidValue;
        switch (p.epi.act) {
        case kActNone: return launch_epi<kActNone>(tile_m, tile_n, map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case kActRelu: return launch_epi<kActRelu>(tile_m, tile_n, map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case kActLeakyRelu: return launch_epi<kActLeakyRelu>(tile_m, tile_n, map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case kActGelu: return launch_epi<kActGelu>(tile_m, tile_n, map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case kActGeluTanh: return launch_epi<kActGeluTanh>(tile_m, tile_n, map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case kActSilu: return launch_epi<kActSilu>(tile_m, tile_n, map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    return launch_plain_or_cluster(tile_m, tile_n, epi, red_cluster, map_a, map_b, map_out, map_ws, map_red,
                                   p, grid, stream);
}

template <int BN>
static cudaError_t capacity_of(int red_cluster, int *clusters)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(red_cluster), 1, 1);
    cfg.blockDim = dim3(gemm_threads(false, true), 1, 1);
    cfg.dynamicSmemBytes = TileCfg<BN, false>::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(red_cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, tsm_gemm_tcgen05_kernel<BN, false, false, true, kActNone>, &cfg);
}

cudaError_t cluster_capacity(int tile_n, int red_cluster, int *clusters)
{
    *clusters = 0;
    cudaError_t e = set_attr<128, false, false, true, kActNone>();
    if (e == cudaSuccess)
        e = set_attr<256, false, false, true, kActNone>();
    if (e != cudaSuccess)
        return e;
    return tile_n == 256 ? capacity_of<256>(red_cluster, clusters) : capacity_of<128>(red_cluster, clusters);
}

cudaError_t launch_splitk_reduce(const float *W, void *C, int32_t M, int32_t N, int32_t S,
                                 int32_t batch, int64_t ldw, int64_t ldc, int64_t strideC,
                                 const Epilogue &epi, int grid, cudaStream_t stream)
{
    tsm_splitk_reduce_kernel<<<grid, 256, 0, stream>>>(W, C, M, N, S, batch, ldw, ldc, strideC, epi);
    return cudaGetLastError();
}

cudaError_t launch_zero_fill(void *C, int32_t M, int32_t N, int32_t batch, int64_t ldc,
                             int64_t strideC, const int32_t *group_rows, const Epilogue &epi,
                             int grid, cudaStream_t stream)
{
    tsm_zero_fill_kernel<<<grid, 256, 0, stream>>>(C, M, N, batch, ldc, strideC, group_rows, epi);
    return cudaGetLastError();
}

namespace {

// Launch shape of a repack: threads per row (a power of two up to 256, enough
// for a row's chunks), chunks per thread per row segment at most 4, and
// enough blocks over the rows to cover the GPU several times.
template <typename T, bool PACK>
cudaError_t launch_repack(const T *src, int64_t s_ld, int64_t s_stride, T *dst, int64_t d_ld,
                          int64_t d_stride, int32_t rows, int32_t cols, int32_t batch,
                          const int32_t *group_rows, int sms, cudaStream_t stream)
{
    constexpr int V = 16 / sizeof(T);
    const int32_t chunks = (cols + V - 1) / V;
    int32_t tpr = 1;
    while (tpr < chunks && tpr < 256)
        tpr *= 2;
    // a segment is a multiple of tpr chunks, at least 4 per thread, and
    // long enough that the segments of a row fit grid.y (65535)
    const int64_t min_seg = (int64_t(chunks) + 65534) / 65535;
    const int32_t seg = int32_t(std::max<int64_t>(int64_t(tpr) * 4, (min_seg + tpr - 1) / tpr * tpr));
    const int32_t rpb = 256 / tpr;
    const int64_t gy = (chunks + int64_t(seg) - 1) / seg;
    const int64_t gz = std::min<int64_t>(batch, 65535);
    const int64_t want = int64_t(sms) * 32;  // blocks in flight over the whole grid
    const int64_t gx = std::max<int64_t>(
        1, std::min<int64_t>((rows + rpb - 1) / rpb, (want + gy * gz - 1) / (gy * gz)));
    tsm_repack_kernel<T, PACK><<<dim3(unsigned(gx), unsigned(gy), unsigned(gz)), 256, 0, stream>>>(
        src, s_ld, s_stride, dst, d_ld, d_stride, rows, cols, batch, tpr, seg, group_rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_f16(const uint16_t *src, int64_t s_ld, int64_t s_stride, uint16_t *dst,
                            int64_t d_ld, int64_t d_stride, int32_t rows, int32_t cols,
                            int32_t batch, int sms, cudaStream_t stream)
{
    return launch_repack<uint16_t, true>(src, s_ld, s_stride, dst, d_ld, d_stride, rows, cols, batch,
                                         nullptr, sms, stream);
}

cudaError_t launch_unpack_f32(const float *src, int64_t s_ld, int64_t s_stride, float *dst,
                              int64_t d_ld, int64_t d_stride, int32_t rows, int32_t cols,
                              int32_t batch, const int32_t *group_rows, int sms,
                              cudaStream_t stream)
{
    return launch_repack<uint32_t, false>(reinterpret_cast<const uint32_t *>(src), s_ld, s_stride,
                                          reinterpret_cast<uint32_t *>(dst), d_ld, d_stride, rows,
                                          cols, batch, group_rows, sms, stream);
}

cudaError_t launch_unpack_u16(const uint16_t *src, int64_t s_ld, int64_t s_stride, uint16_t *dst,
                              int64_t d_ld, int64_t d_stride, int32_t rows, int32_t cols,
                              int32_t batch, const int32_t *group_rows, int sms,
                              cudaStream_t stream)
{
    return launch_repack<uint16_t, false>(src, s_ld, s_stride, dst, d_ld, d_stride, rows, cols, batch,
                                          group_rows, sms, stream);
}

cudaError_t device_status_word(uint32_t **ptr)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_status_word);
}

}  // namespace tsm
