// rowsum_kernels.cu -- the tiled row sum and the GEMV (N = 1): memory-bound
// reductions along a row with a deterministic, fixed-order reduce.
//
// The row sum is the kernel of "A Dumb Triton Runtime Error" ("The kernel
// itself"): out[r] = sum over c < C of x[r * row_stride + c * col_stride], the
// elements widened to f32 and accumulated in f32, the lanes' partial sums
// combined by a tree on the chip rather than by atomics onto the output (the
// page's closing section: atomics accumulate onto whatever is in out, and
// their order is not fixed).  The GEMV is the same walk over a row of A with
// each element multiplied by x[k] first.
//
// A worker is `tpr` consecutive lanes of a warp (a power of two up to 32).
// It reduces one item -- row r, columns [s * seg, min(C, (s + 1) * seg)) --
// each lane taking every tpr-th 16-byte chunk (or element) of the segment
// into eight (four) accumulators in turn -- that many loads in flight --,
// then the accumulators in a fixed order, then a butterfly
// over the worker's lanes.  With one segment per row the sum goes straight
// to out[r]; otherwise to partial[r * segs + s], summed over s in ascending
// order by a second kernel.  The order depends only on (R, C) and the launch
// shape the host derives from them, so a call is bitwise reproducible.
#include "gemm_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tsm {

namespace {

// Element types: 0 f32, 1 f16 (IEEE binary16), 2 bf16 (upper half of a binary32).
template <int ET>
__device__ __forceinline__ float elem_f32(uint32_t bits)
{
    if constexpr (ET == kOutF16)
        return __half2float(__ushort_as_half(uint16_t(bits)));
    else if constexpr (ET == kOutBF16)
        return __uint_as_float(bits << 16);
    else
        return __uint_as_float(bits);
}

// The sum of one 16-byte chunk (8 16-bit or 4 f32 values), pairwise in a
// fixed order; with GEMV the products with the matching chunk of x.
template <int ET, bool GEMV>
__device__ __forceinline__ float chunk_sum(const uint4 &a, const uint4 &x)
{
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
    float s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (ET == kOutF32) {
            s[i] = GEMV ? 0.f : __uint_as_float(w[i]);
        } else {
            const float lo = elem_f32<ET>(w[i] & 0xffffu), hi = elem_f32<ET>(w[i] >> 16);
            if constexpr (GEMV) {
                const float xl = elem_f32<kOutF16>(xv[i] & 0xffffu), xh = elem_f32<kOutF16>(xv[i] >> 16);
                s[i] = fmaf(hi, xh, lo * xl);
            } else {
                s[i] = lo + hi;
            }
        }
    }
    return (s[0] + s[1]) + (s[2] + s[3]);
}

}  // namespace

template <int ET, bool VEC, bool GEMV>
__global__ void __launch_bounds__(256) tsm_row_reduce_kernel(RowReduceParams p)
{
    constexpr int EB = ET == kOutF32 ? 4 : 2;  // element bytes
    constexpr int V = 16 / EB;                  // elements per 16-byte chunk
    const int lane = int(threadIdx.x & 31);
    const int tpr = p.tpr;
    const int sub = lane & (tpr - 1);
    const int64_t per_warp = 32 / tpr;
    const int64_t warp = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int64_t workers = int64_t(gridDim.x) * (blockDim.x / 32) * per_warp;
    const int64_t items = p.R * p.segs;
    const char *X = static_cast<const char *>(p.X);
    // Every lane of a warp runs the same number of passes (the shuffles need
    // them all); a worker past the last item adds nothing and stores nothing.
    for (int64_t first = warp * per_warp; first < items; first += workers) {
        const int64_t q = first + lane / tpr;
        const bool active = q < items;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float tail = 0.f;
        if (active) {
            const int64_t r = q / p.segs;
            const int64_t s = q - r * p.segs;
            const int64_t c0 = s * p.seg;
            const int64_t c1 = min(p.C, c0 + p.seg);
            if constexpr (VEC) {
                // c0 is a multiple of V (seg is); whole chunks, then < V elements.
                const char *row = X + (r * p.row_stride + c0) * EB;
                const int64_t nchunk = (c1 - c0) / V;
                const uint4 *ap = reinterpret_cast<const uint4 *>(row);
                const uint4 *xp = GEMV ? reinterpret_cast<const uint4 *>(p.xv + c0) : nullptr;
                if constexpr (ET == kOutF32) {
                    // Whole groups of eight independent loads, then the last,
                    // partial group (chunk k + j * tpr still to acc[j]).
                    // For f32 this form keeps eight loads in flight (1.3-1.9x
                    // faster on GB300, 55 registers instead of 74); for the
                    // 16-bit types the guarded form below measured faster.
                    int64_t k = sub;
                    for (; k + 7 * int64_t(tpr) < nchunk; k += 8 * tpr) {
                        uint4 a[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            a[j] = __ldg(ap + k + int64_t(j) * tpr);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            acc[j] += chunk_sum<ET, false>(a[j], a[j]);
                    }
#pragma unroll
                    for (int j = 0; j < 7; ++j)
                        if (k + int64_t(j) * tpr < nchunk) {
                            const uint4 aj = __ldg(ap + k + int64_t(j) * tpr);
                            acc[j] += chunk_sum<ET, false>(aj, aj);
                        }
                } else {
                for (int64_t k = sub; k < nchunk; k += 8 * tpr) {
                        uint4 a[8], xv[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int64_t kk = k + int64_t(j) * tpr;
                            if (kk < nchunk) {
                                a[j] = __ldg(ap + kk);
                                if constexpr (GEMV)
                                    xv[j] = __ldg(xp + kk);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (k + int64_t(j) * tpr < nchunk)
                                acc[j] += chunk_sum<ET, GEMV>(a[j], GEMV ? xv[j] : a[j]);
                    }
                }
                if (sub == 0) {
                    for (int64_t c = c0 + nchunk * V; c < c1; ++c) {
                        uint32_t bits;
                        if constexpr (EB == 4)
                            bits = __ldg(reinterpret_cast<const uint32_t *>(X) + r * p.row_stride + c);
                        else
                            bits = __ldg(reinterpret_cast<const uint16_t *>(X) + r * p.row_stride + c);
                        float v = elem_f32<ET>(bits);
                        if constexpr (GEMV)
                            v *= __half2float(__ushort_as_half(__ldg(p.xv + c * p.incx)));
                        tail += v;
                    }
                }
            } else {
                for (int64_t c = c0 + sub; c < c1; c += 4 * tpr) {
                    float v[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int64_t cc = c + int64_t(j) * tpr;
                        v[j] = 0.f;
                        if (cc < c1) {
                            const int64_t at = r * p.row_stride + cc * p.col_stride;
                            uint32_t bits;
                            if constexpr (EB == 4)
                                bits = __ldg(reinterpret_cast<const uint32_t *>(X) + at);
                            else
                                bits = __ldg(reinterpret_cast<const uint16_t *>(X) + at);
                            v[j] = elem_f32<ET>(bits);
                            if constexpr (GEMV)
                                v[j] *= __half2float(__ushort_as_half(__ldg(p.xv + cc * p.incx)));
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        acc[j] += v[j];
                }
            }
        }
        float v = (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]))) + tail;
        for (int o = tpr >> 1; o >= 1; o >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, o);
        if (active && sub == 0) {
            if (p.segs == 1)
                p.out[q] = v;
            else
                p.partial[q] = v;
        }
    }
}

// out[r] from the segs partial sums of row r, one warp per row: lane l adds
// partials l, l + 32, l + 64, ... in ascending order, then the lanes' sums
// meet in a fixed butterfly -- a fixed order, so the result is reproducible.
__global__ void __launch_bounds__(256) tsm_row_partials_kernel(const float *__restrict__ partial,
                                                               float *__restrict__ out, int64_t R,
                                                               int32_t segs)
{
    const int lane = int(threadIdx.x & 31);
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x / 32);
    for (int64_t r = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5); r < R; r += warps) {
        const float *pr = partial + r * segs;
        float v = 0.f;
        int32_t s = lane;
        // Eight loads in flight, added in the same ascending order.
        for (; s + 7 * 32 < segs; s += 8 * 32) {
            float t[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                t[j] = pr[s + 32 * j];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v += t[j];
        }
        for (; s < segs; s += 32)
            v += pr[s];
        for (int o = 16; o >= 1; o >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0)
            out[r] = v;
    }
}

template <int ET, bool GEMV>
static cudaError_t launch_et(const RowReduceParams &p, bool vec, int grid, cudaStream_t stream)
{
    if (vec)
        tsm_row_reduce_kernel<ET, true, GEMV><<<grid, 256, 0, stream>>>(p);
    else
        tsm_row_reduce_kernel<ET, false, GEMV><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int ET, bool GEMV>
static int blocks_et(bool vec)
{
    int n = 0;
    cudaError_t e = vec ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                              &n, tsm_row_reduce_kernel<ET, true, GEMV>, 256, 0)
                        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                              &n, tsm_row_reduce_kernel<ET, false, GEMV>, 256, 0);
    return e == cudaSuccess && n > 0 ? n : 1;
}

int row_reduce_blocks_per_sm(int elem, bool vec, bool gemv)
{
    if (gemv)
        return blocks_et<kOutF16, true>(vec);
    switch (elem) {
    case kOutF32: return blocks_et<kOutF32, false>(vec);
    case kOutF16: return blocks_et<kOutF16, false>(vec);
    default: return blocks_et<kOutBF16, false>(vec);
    }
}

cudaError_t launch_row_reduce(const RowReduceParams &p, int elem, bool vec, bool gemv, int grid,
                              cudaStream_t stream)
{
    if (gemv)
        return launch_et<kOutF16, true>(p, vec, grid, stream);
    switch (elem) {
    case kOutF32: return launch_et<kOutF32, false>(p, vec, grid, stream);
    case kOutF16: return launch_et<kOutF16, false>(p, vec, grid, stream);
    case kOutBF16: return launch_et<kOutBF16, false>(p, vec, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_row_partials(const float *partial, float *out, int64_t R, int32_t segs, int grid,
                                cudaStream_t stream)
{
    tsm_row_partials_kernel<<<grid, 256, 0, stream>>>(partial, out, R, segs);
    return cudaGetLastError();
}

}  // namespace tsm
