// gemm_epi.cu -- the GEMM kernels with a fused epilogue for one activation,
// TSM_EPI_ACT (one of the kAct* values): one CTA per tile (64, 128 or 256
// columns) and CTA pairs (128 or 256).  The build compiles this unit once per
// activation, in parallel, so that each kernel holds only its own
// activation's code and the units stay small.
#include "gemm_kernel.cuh"

#ifndef TSM_EPI_ACT
#error "compile with -DTSM_EPI_ACT=<activation>"
#endif

namespace tsm {

template <int ACT>
cudaError_t set_epi_attributes(int tile_m, int tile_n)
{
    if (tile_m == 2 * kTileM) {
        switch (tile_n) {
        case 128: return set_attr<128, true, true, false, ACT>();
        case 256: return set_attr<256, true, true, false, ACT>();
        case 512: return set_attr<512, true, true, false, ACT>();
        default: return cudaErrorInvalidValue;
        }
    }
    switch (tile_n) {
    case 64: return set_attr<64, false, true, false, ACT>();
    case 128: return set_attr<128, false, true, false, ACT>();
    case 256: return set_attr<256, false, true, false, ACT>();
    default: return cudaErrorInvalidValue;
    }
}

template <int ACT>
cudaError_t launch_epi(int tile_m, int tile_n, const CUtensorMap &map_a, const CUtensorMap &map_b,
                       const CUtensorMap &map_out, const CUtensorMap &map_ws, const CUtensorMap &map_red,
                       const KernelParams &p, int grid, cudaStream_t stream)
{
    if (tile_m == 2 * kTileM) {
        switch (tile_n) {
        case 128: return launch_bn<128, true, true, false, ACT>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case 256: return launch_bn<256, true, true, false, ACT>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        case 512: return launch_bn<512, true, true, false, ACT>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (tile_n) {
    case 64: return launch_bn<64, false, true, false, ACT>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
    case 128: return launch_bn<128, false, true, false, ACT>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
    case 256: return launch_bn<256, false, true, false, ACT>(map_a, map_b, map_out, map_ws, map_red, p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

template cudaError_t set_epi_attributes<TSM_EPI_ACT>(int, int);
template cudaError_t launch_epi<TSM_EPI_ACT>(int, int, const CUtensorMap &, const CUtensorMap &,
                                             const CUtensorMap &, const CUtensorMap &, const CUtensorMap &,
                                             const KernelParams &, int, cudaStream_t);

}  // namespace tsm
