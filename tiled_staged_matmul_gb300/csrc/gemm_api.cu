// gemm_api.cu -- host side of the C ABI declared in include/tsm_gemm.h:
// argument checks, the planner (tile width, ring depth, split-K factor,
// grid), tensor-map encoding, the split-K workspace and the launches.
//
// The planner is the GB300 counterpart of the pages' footprint check and
// K_TILE choice ("The PTSS Cliff: A Kernel That Won't Build", sections "The
// SLM Footprint", "Choosing K_TILE" and "The Four Gates"): the K depth of a
// staged block is fixed at 64 (one 128-byte swizzle row of f16), the ring
// takes as many A+B blocks as fit the 227 KiB shared-memory budget next to
// the epilogue's staging buffers, and the tile width and split factor are
// chosen so that the persistent grid fills the SMs.  Unlike the pages' pass
// there is no "decline" outcome: ragged K is handled by zero fill rather
// than by a divisibility gate.
#include "../../include/tsm_gemm.h"
#include "gemm_internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace tsm {
namespace {

thread_local std::string g_last_error;

// A 64-bit value unique to each launch of this process (a bijective mix of a
// per-process start value and a call counter), never 0, and unlikely to
// equal any word another process or earlier data left in recycled memory.
uint64_t next_launch_epoch()
{
    static const uint64_t start = uint64_t(std::chrono::steady_clock::now().time_since_epoch().count()) ^
                                  (uint64_t(reinterpret_cast<uintptr_t>(&g_last_error)) << 17);
    static std::atomic<uint64_t> calls{0};
    for (;;) {
        uint64_t z = start + 0x9e3779b97f4a7c15ull * (calls.fetch_add(1) + 1);
        z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
        z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
        z ^= z >> 31;
        if (z != 0)
            return z;
    }
}

gemm_status_t fail(gemm_status_t st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

gemm_status_t fail_cuda(cudaError_t e, const char *what)
{
    return fail(GEMM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
// Dynamic shared memory of a GEMM CTA outside its operand ring and epilogue
// buffers: the alignment slack and the control block (TileCfg).
constexpr int64_t kSmemSlackAndControl = 1024 + 2048;
constexpr int64_t kInt32Max = 2147483647;

// ------------------------------------------------------------- driver entry points

struct Driver {
    PFN_cuTensorMapEncodeTiled_v12000 encode_tiled = nullptr;
    PFN_cuPointerGetAttributes_v7000 pointer_attributes = nullptr;
    bool loaded = false;
    std::string error;
};

Driver &driver()
{
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound;
        cudaDriverEntryPointQueryResult q2 = cudaDriverEntryPointSymbolNotFound;
        void *f1 = nullptr, *f2 = nullptr;
        cudaError_t e1 =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000, cudaEnableDefault, &q1);
        cudaError_t e2 =
            cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &f2, 12000, cudaEnableDefault, &q2);
        if (e1 != cudaSuccess || q1 != cudaDriverEntryPointSuccess || !f1) {
            d.error = "cuTensorMapEncodeTiled is not available from the driver";
            return;
        }
        d.encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f1);
        if (e2 != cudaSuccess || q2 != cudaDriverEntryPointSuccess || !f2) {
            d.error = "cuPointerGetAttributes is not available from the driver";
            return;
        }
        d.pointer_attributes = reinterpret_cast<PFN_cuPointerGetAttributes_v7000>(f2);
        d.loaded = true;
    });
    return d;
}

// ------------------------------------------------------------- per-device state

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    int smem_optin = 0;
    bool attrs_set[46] = {};  // see attr_index
    cudaMemPool_t pool = nullptr;
    uint32_t *status = nullptr;
    // Clusters of 2 and of 4 CTAs of the cluster-sum kernel that fit at once.
    int caps2 = 0, caps4 = 0;
};

DeviceState g_devices[kMaxDevices];
std::mutex g_device_mutex;

gemm_status_t device_state(int dev, DeviceState **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GEMM_ERR_INVALID_VALUE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_device_mutex);
    DeviceState &s = g_devices[dev];
    if (!s.ready) {
        cudaError_t e;
        if ((e = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
        cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&s.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (s.cc_major != 10 || s.cc_minor != 3)
            return fail(GEMM_ERR_UNSUPPORTED_DEVICE,
                        "device %d has compute capability %d.%d; this library is built for 10.3 "
                        "(GB300, sm_103a) only",
                        dev, s.cc_major, s.cc_minor);
        if ((e = device_status_word(&s.status)) != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(status word)");
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if ((e = cudaMemPoolCreate(&s.pool, &props)) != cudaSuccess)
            return fail_cuda(e, "cudaMemPoolCreate(split-K workspace pool)");
        uint64_t keep = UINT64_MAX;  // keep freed workspace for the next call
        cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep);
        // Every CTA of an in-kernel split-K sum must be resident at once (they
        // wait for one another), so the cluster sum is planned only within
        // what the occupancy API says fits.
        if ((e = cluster_capacity(128, 2, &s.caps2)) != cudaSuccess ||
            (e = cluster_capacity(128, 4, &s.caps4)) != cudaSuccess)
            return fail_cuda(e, "cudaOccupancyMaxActiveClusters(cluster split-K sum)");
        s.ready = true;
    }
    *out = &s;
    return GEMM_OK;
}

// One slot per kernel instantiation: single-CTA tile_n 64 / 128 / 256, CTA-pair 128 / 256.
int config_index(int tile_m, int tile_n)
{
    if (tile_m == 2 * kTileM)
        return tile_n == 128 ? 3 : 4;
    return tile_n == 64 ? 0 : tile_n == 128 ? 1 : 2;
}

// Slot of DeviceState::attrs_set: the plain kernels 0-4, with the fused
// epilogue 5-34 (five tile shapes for each of the six activations), the
// cluster-sum kernels (tile_n 128 / 256, plain or fused) 35-38, the
// 256 x 512 pair tile 39 (plain) and 40-45 (fused, one per activation).
int attr_index(int tile_m, int tile_n, bool epi, int red_cluster, int act)
{
    if (tile_n == 512)
        return epi ? 40 + act : 39;
    if (red_cluster > 1)
        return 35 + (tile_n == 256 ? 1 : 0) + (epi ? 2 : 0);
    return config_index(tile_m, tile_n) + (epi ? 5 + 5 * act : 0);
}

// Estimated clusters of `n` CTAs (one per SM) that fit at once on a GB300 of
// `sms` SMs, for planning without a device: pairs fit everywhere; four-CTA
// clusters leave the SMs of each GPC past a multiple of four idle (36 of 38
// on the 152-SM part, as the occupancy API reports there).
int estimated_cluster_capacity(int sms, int n)
{
    return n == 2 ? sms / 2 : sms / 4 * 18 / 19;
}

// ------------------------------------------------------------- argument checks

struct Problem {
    const uint16_t *A;
    const uint16_t *B;
    void *C;  // epi.out_type elements
    int64_t M, N, K, lda, ldb, ldc, sA, sB, sC, batch;
    // Grouped launch (at most kMaxGroupsPerLaunch groups = batches): device
    // array of each group's row count; null for plain and batched GEMMs.
    const int32_t *group_rows = nullptr;
    // What the kernels do to each output value before storing it.
    Epilogue epi;
};

// Bytes spanned by `batch` matrices of `rows` x `cols` elements of `elem`
// bytes, row stride `ld`, batch stride `stride` (all in elements).
int64_t span_bytes(int64_t batch, int64_t stride, int64_t rows, int64_t ld, int64_t cols, int64_t elem)
{
    if (batch <= 0 || rows <= 0 || cols <= 0)
        return 0;
    return ((batch - 1) * stride + (rows - 1) * ld + cols) * elem;
}

bool overlaps(const void *p, int64_t pn, const void *q, int64_t qn)
{
    if (pn <= 0 || qn <= 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), a1 = a0 + uint64_t(pn);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(q), b1 = b0 + uint64_t(qn);
    return a0 < b1 && b0 < a1;
}

// Checks that need no GPU.  Sets *trivial when there is nothing to compute.
gemm_status_t check_host(const Problem &pr, bool *trivial)
{
    *trivial = false;
    if (pr.M < 0 || pr.N < 0 || pr.K < 0 || pr.batch < 0)
        return fail(GEMM_ERR_INVALID_VALUE, "negative size: M=%lld N=%lld K=%lld batch=%lld",
                    (long long)pr.M, (long long)pr.N, (long long)pr.K, (long long)pr.batch);
    if (pr.M > kInt32Max || pr.N > kInt32Max || pr.K > kInt32Max || pr.batch > kInt32Max)
        return fail(GEMM_ERR_INVALID_VALUE, "M, N, K and batch must be below 2^31");
    if (pr.M == 0 || pr.N == 0 || pr.batch == 0) {
        *trivial = true;
        return GEMM_OK;
    }
    if (!pr.C)
        return fail(GEMM_ERR_INVALID_VALUE, "C is NULL");
    if (pr.ldc < pr.N)
        return fail(GEMM_ERR_INVALID_VALUE, "ldc (%lld) < N (%lld)", (long long)pr.ldc, (long long)pr.N);
    if (pr.K > 0) {
        if (!pr.A || !pr.B)
            return fail(GEMM_ERR_INVALID_VALUE, "A or B is NULL");
        if (pr.lda < pr.K)
            return fail(GEMM_ERR_INVALID_VALUE, "lda (%lld) < K (%lld)", (long long)pr.lda, (long long)pr.K);
        if (pr.ldb < pr.N)
            return fail(GEMM_ERR_INVALID_VALUE, "ldb (%lld) < N (%lld)", (long long)pr.ldb, (long long)pr.N);
    }
    if (pr.batch > 1 && (pr.sC <= 0 || (pr.K > 0 && (pr.sA <= 0 || pr.sB <= 0))))
        return fail(GEMM_ERR_INVALID_VALUE, "batch strides must be positive when batch > 1");
    // Every element at its natural alignment (any pitch is fine: an operand
    // the TMA cannot address is repacked, see run_repacked).
    const int eb = pr.epi.out_bytes();
    if (reinterpret_cast<uintptr_t>(pr.C) & uintptr_t(eb - 1))
        return fail(GEMM_ERR_MISALIGNED, "C must be %d-byte aligned (its elements)", eb);
    if (pr.K > 0 && ((reinterpret_cast<uintptr_t>(pr.A) & 1u) || (reinterpret_cast<uintptr_t>(pr.B) & 1u)))
        return fail(GEMM_ERR_MISALIGNED, "A and B must be 2-byte aligned (f16 elements)");
    if (pr.batch > 1 && pr.sC < (pr.M - 1) * pr.ldc + pr.N)
        return fail(GEMM_ERR_ALIAS, "batches of C overlap (strideC too small)");
    const int64_t bytesC = span_bytes(pr.batch, pr.sC, pr.M, pr.ldc, pr.N, eb);
    if (pr.epi.bias) {
        if (reinterpret_cast<uintptr_t>(pr.epi.bias) & 3u)
            return fail(GEMM_ERR_MISALIGNED, "bias must be 4-byte aligned (f32)");
        if (pr.epi.bias_stride < 0)
            return fail(GEMM_ERR_INVALID_VALUE, "bias_stride must be >= 0");
        const int64_t bytesBias = span_bytes(pr.batch, pr.epi.bias_stride, 1, pr.N, pr.N, 4);
        if (overlaps(pr.C, bytesC, pr.epi.bias, bytesBias))
            return fail(GEMM_ERR_ALIAS, "C overlaps the bias");
    }
    if (pr.K > 0) {
        const int64_t bytesA = span_bytes(pr.batch, pr.sA, pr.M, pr.lda, pr.K, 2);
        const int64_t bytesB = span_bytes(pr.batch, pr.sB, pr.K, pr.ldb, pr.N, 2);
        if (overlaps(pr.C, bytesC, pr.A, bytesA) || overlaps(pr.C, bytesC, pr.B, bytesB))
            return fail(GEMM_ERR_ALIAS, "C overlaps A or B");
    }
    return GEMM_OK;
}

// What the tensor-memory accelerator can address: a 16-byte aligned base and
// row / batch pitches that are multiples of 16 bytes ("Intel XPU Backend for
// Triton", section "Use Tensor Descriptors to load tl.dot arguments and save
// results": a descriptor wants its last stride 1 and the others aligned).
struct TmaLayout {
    bool a, b, c;
    bool all() const { return a && b && c; }
};

TmaLayout tma_layout(const Problem &pr)
{
    TmaLayout t;
    const int64_t per16 = 16 / pr.epi.out_bytes();  // C elements per 16 bytes
    t.c = !((reinterpret_cast<uintptr_t>(pr.C) & 15u) || (pr.ldc % per16) ||
            (pr.batch > 1 && pr.sC % per16));
    t.a = pr.K == 0 ||
          !((reinterpret_cast<uintptr_t>(pr.A) & 15u) || (pr.lda % 8) || (pr.batch > 1 && pr.sA % 8));
    t.b = pr.K == 0 ||
          !((reinterpret_cast<uintptr_t>(pr.B) & 15u) || (pr.ldb % 8) || (pr.batch > 1 && pr.sB % 8));
    return t;
}

// The pointer is device memory of `dev` and its allocation covers `bytes`:
// one driver query for the memory type, the managed flag, the device and the
// allocation's range (a pointer the driver does not know comes back as type 0).
gemm_status_t check_device_pointer(const void *p, int64_t bytes, int dev, const char *name)
{
    Driver &d = driver();
    if (!d.loaded)
        return fail(GEMM_ERR_CUDA, "%s", d.error.c_str());
    unsigned int type = 0, managed = 0;
    int ordinal = -1;
    CUdeviceptr start = 0;
    size_t size = 0;
    CUpointer_attribute attrs[5] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_IS_MANAGED,
                                    CU_POINTER_ATTRIBUTE_DEVICE_ORDINAL, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR,
                                    CU_POINTER_ATTRIBUTE_RANGE_SIZE};
    void *data[5] = {&type, &managed, &ordinal, &start, &size};
    const CUresult r = d.pointer_attributes(5, attrs, data, CUdeviceptr(reinterpret_cast<uintptr_t>(p)));
    if (r != CUDA_SUCCESS)
        return fail(GEMM_ERR_INVALID_VALUE, "%s: the driver cannot query the pointer (CUresult %d)", name, int(r));
    if (type != CU_MEMORYTYPE_DEVICE && !managed)
        return fail(GEMM_ERR_INVALID_VALUE, type == 0 ? "%s is not a CUDA pointer" : "%s is not device memory", name);
    if (ordinal != dev)
        return fail(GEMM_ERR_INVALID_VALUE, "%s lives on device %d, the current device is %d", name, ordinal, dev);
    if (size > 0) {
        const uint64_t end = uint64_t(reinterpret_cast<uintptr_t>(p)) + uint64_t(bytes);
        if (end > uint64_t(start) + uint64_t(size))
            return fail(GEMM_ERR_INVALID_VALUE,
                        "%s: the allocation ends %llu bytes before the last element", name,
                        (unsigned long long)(end - (uint64_t(start) + uint64_t(size))));
    }
    return GEMM_OK;
}

// ------------------------------------------------------------- planner

int ceil_div(int64_t a, int64_t b) { return int((a + b - 1) / b); }

// Candidate tile shapes, in the order ties are broken (a CTA pair per
// 256-row tile halves each SM's B traffic).
struct TileChoice {
    int tile_m, tile_n;
};
// The 256 x 512 pair tile (one accumulator, two 256-column MMAs per k-step
// on one A tile) takes whole tiles only: no K split, no tail.
constexpr TileChoice kChoices[] = {{256, 256}, {256, 128}, {128, 256}, {128, 128}, {128, 64}, {256, 512}};

// `wide`: the planner may pick the 256 x 512 tile by itself (it is always
// taken when asked for).
gemm_status_t make_plan(int64_t M, int64_t N, int64_t K, int64_t batch, const gemm_options_t *o,
                        int sms, int caps2, int caps4, gemm_plan_info_t *pl, bool wide)
{
    if (sms <= 0)
        return fail(GEMM_ERR_INVALID_VALUE, "SM count must be positive");
    memset(pl, 0, sizeof *pl);
    const int req_n = o ? o->tile_n : 0;
    const int req_m = o ? o->tile_m : 0;
    if (req_n != 0 && req_n != 64 && req_n != 128 && req_n != 256 && req_n != 512)
        return fail(GEMM_ERR_INVALID_VALUE, "tile_n must be 0, 64, 128, 256 or 512 (got %d)", req_n);
    if (req_m != 0 && req_m != 128 && req_m != 256)
        return fail(GEMM_ERR_INVALID_VALUE, "tile_m must be 0, 128 or 256 (got %d)", req_m);
    if (req_m == 256 && req_n == 64)
        return fail(GEMM_ERR_INVALID_VALUE, "tile_m 256 (a CTA pair) needs tile_n 128, 256 or 512");
    if (req_n == 512 && req_m == 128)
        return fail(GEMM_ERR_INVALID_VALUE, "tile_n 512 is a CTA pair's tile: tile_m must be 0 or 256");
    if (req_n == 512 && o && o->split_k > 1)
        return fail(GEMM_ERR_INVALID_VALUE, "tile_n 512 takes whole tiles: split_k must be 0 or 1");
    if (req_n == 512 && sms < 2)
        return fail(GEMM_ERR_INVALID_VALUE, "a CTA pair needs at least two SMs");
    if (req_m == 256 && sms < 2)
        return fail(GEMM_ERR_INVALID_VALUE, "a CTA pair needs at least two SMs");
    const int req_s = o ? o->split_k : 0;
    if (req_s < 0)
        return fail(GEMM_ERR_INVALID_VALUE, "split_k must be >= 0");
    if (o && (o->splitk_reduce < 0 || o->splitk_reduce > 2))
        return fail(GEMM_ERR_INVALID_VALUE, "splitk_reduce must be 0, 1 or 2");
    if (o && (o->split_tail < 0 || o->split_tail > 3))
        return fail(GEMM_ERR_INVALID_VALUE, "split_tail must be 0, 1, 2 or 3");
    const int req_c = o ? o->red_cluster : 0;
    if (req_c != 0 && req_c != 1 && req_c != 2 && req_c != 4)
        return fail(GEMM_ERR_INVALID_VALUE, "red_cluster must be 0, 1, 2 or 4 (got %d)", req_c);
    const int k_blocks = ceil_div(std::max<int64_t>(K, 1), kTileK);
    const int64_t Mx = std::max<int64_t>(M, 1), Nx = std::max<int64_t>(N, 1);
    const int64_t ldw = (N + 3) / 4 * 4;
    auto tiles_of = [&](int tm, int tn) { return int64_t(ceil_div(Mx, tm)) * ceil_div(Nx, tn) * batch; };
    auto slots_of = [&](int tm) { return int64_t(tm == 2 * kTileM ? sms / 2 : sms); };
    auto tile_elems_of = [](int tm, int tn) { return int64_t(tm) * tn; };
    // The planner's own pick of the 256 x 512 tile: only where no K split
    // and no tail are asked for, since that tile takes neither.
    const int req_tail = o ? o->split_tail : 0;
    const bool wide_auto = wide && req_s <= 1 && req_tail != 1 && req_tail != 3;
    auto allowed = [&](const TileChoice &c) {
        return (req_m == 0 || req_m == c.tile_m) &&
               (req_n == 0 ? wide_auto || c.tile_n != 512 : req_n == c.tile_n) &&
               (c.tile_m == kTileM || sms >= 2);
    };
    // K ranges that put about one unit on every slot, at least 4 k-blocks each.
    auto split_for = [&](int tm, int tn) -> int {
        if (tn == 512)
            return 1;
        if (req_s > 0)
            return std::min(req_s, k_blocks);
        const int64_t tiles = tiles_of(tm, tn);
        if (K == 0 || tiles >= slots_of(tm))
            return 1;
        return int(std::max<int64_t>(1, std::min<int64_t>(slots_of(tm) / tiles, k_blocks / 4)));
    };
    // Tail of a plan with more tiles than slots whose last wave is at most
    // half full (gemm_options_t.split_tail: 0 auto, 1 K ranges, 2 none,
    // 3 column slices).  Either each of the R tiles of that wave is split
    // into `pieces` K ranges summed in the kernel, or it is cut into `pieces`
    // column slices computed over all of K (no partial sums, any batch).
    // `frac` is the time of the last wave in whole-tile times.
    struct Tail {
        int pieces = 0;
        bool narrow = false;
        double frac = 1.0;
    };
    // One CTA's time per k-block of a unit `w` columns wide (us): its MMAs at
    // ~13.1 TFLOP/s per SM, or bringing its A and B boxes into shared memory
    // at ~87 GB/s per SM, whichever is longer (measured on GB300: 256 x 256
    // pair tiles run ~15 % over their MMA time, 256 x 128 column slices at
    // three quarters of a whole tile's time).
    // The 256 x 512 pair tile: its MMAs at ~12.5 TFLOP/s per SM (measured
    // on GB300 at 8192^3 and 6144^3; a quarter fewer operand bytes per flop
    // than 256 x 256, so the MMAs bound it).
    auto kb_us = [&](int tm, int w) {
        if (w == 512)
            return 2.0 * kTileM * w * kTileK / 12.5e12 * 1e6;
        const double mma = 2.0 * kTileM * w * kTileK / 13.1e12 * 1e6;
        const double bytes = 2.0 * kTileK * (kTileM + (tm == 2 * kTileM ? w / 2 : w));
        return std::max(mma, bytes / 87e9 * 1e6);
    };
    auto tail_of = [&](int tm, int tn) -> Tail {
        const int mode = o ? o->split_tail : 0;
        const int req_r0 = o ? o->splitk_reduce : 0;
        Tail none;
        if (mode == 2 || req_s != 0 || K == 0 || tn == 512)
            return none;
        const int64_t slots = slots_of(tm), tiles = tiles_of(tm, tn);
        const int64_t rem = tiles % slots;
        if (tiles <= slots || rem == 0)
            return none;
        const double tile_us = double(k_blocks) * kb_us(tm, tn);
        Tail ks;  // K ranges: storing and summing the partials costs about 6 us (measured)
        if (mode != 3 && req_r0 != 1 && batch == 1) {
            const int64_t st = std::min<int64_t>(slots / rem, k_blocks / 4);
            const int64_t reducers = st * (tm == 2 * kTileM ? 2 : 1);
            const int64_t rows_per = (tm + reducers - 1) / reducers;
            const SmemBudget b = smem_budget(tm, tn);
            if (st >= 2 && st <= 256 && rows_per * tn * 4 * st <= int64_t(b.stages) * b.stage_bytes)
                ks = Tail{int(st), false, 1.0 / double(st) + 6.0 / tile_us};
        }
        Tail ns;  // column slices of at least 64 columns of B per CTA
        if (mode != 1) {
            const int b_cols = tm == 2 * kTileM ? tn / 2 : tn;
            int n = 1;
            while (n * 2 <= b_cols / 64 && rem * n * 2 <= slots)
                n *= 2;
            if (n >= 2)
                ns = Tail{n, true, kb_us(tm, tn / n) / kb_us(tm, tn)};
        }
        if (mode == 1)
            return ks;
        if (mode == 3)
            return ns;
        // Auto: the fastest last wave, measured on GB300 in interleaved runs
        // against whole tiles: K ranges x2.0 at 2304 x 2304 x 8192, +2.6 %
        // at 8192^3, +6 % at 5120^3; column slices +25 % at 2304 x 2304 x
        // 1024, +5 % at 4096^2 x 1024, +2 % at 8192^2 x 2048.
        Tail best = none;
        if (ks.pieces && ks.frac < best.frac)
            best = ks;
        if (ns.pieces && ns.frac < best.frac)
            best = ns;
        return best;
    };
    // Long K on a small output: the split-K regime (costed below by per-SM
    // time, partial sums included).
    const bool long_k = req_s == 0 && K > 0 && k_blocks >= 16 &&
                        tiles_of(2 * kTileM, 256) * 2 <= slots_of(2 * kTileM);
    const TileChoice *best = nullptr;
    double best_cost = 0;
    for (const TileChoice &c : kChoices) {
        if (!allowed(c))
            continue;
        const int64_t tiles = tiles_of(c.tile_m, c.tile_n);
        double cost;
        if (long_k) {
            // Each unit's K range at the tile's time per k-block, in waves of
            // units; split partials cost ~2 us plus ~20 us per MB each CTA
            // stores (and its reducer rows read back); pairs their fixed
            // ~8 us.  Fitted to every tile shape timed on 44 long-K shapes on
            // GB300: within 0.1 % (geometric mean) of the fastest, against
            // 4.2 % for a count of bytes moved; on 256 x 256 x 65536 it keeps
            // 128 x 128 tiles in 38 splits (27.7 us; 128 x 256 in 76: 29.7).
            const int sk = split_for(c.tile_m, c.tile_n);
            const int64_t units = tiles * sk;
            const int64_t waves = (units + slots_of(c.tile_m) - 1) / slots_of(c.tile_m);
            const double partial_mb = 2.0 * kTileM * c.tile_n * 4 / 1e6;
            cost = double(waves) * ceil_div(k_blocks, sk) * kb_us(c.tile_m, c.tile_n) +
                   (sk > 1 ? 2.0 + 20.0 * partial_mb : 0.0) + (c.tile_m == 2 * kTileM ? 8.0 : 0.0);
        } else {
            // Full waves of persistent CTAs at the tile's time per k-block
            // (kb_us), and the last wave: whole, or spread over every slot by
            // the tail that tail_of picks for this tile.  CTA pairs carry a
            // fixed ~8 us more: measured on GB300 they are 2-8 us slower than
            // one CTA per tile where both take the same time per k-block
            // (19.6 against 12.3 us at 1024 x 1024 x 512), and with 8 us this
            // choice came within 0.4 % (geometric mean) of the fastest tile on
            // 156 timed shapes.
            const int64_t slots = slots_of(c.tile_m);
            const Tail tl = tail_of(c.tile_m, c.tile_n);
            const double waves = tl.pieces ? double(tiles / slots) + tl.frac
                                           : double((tiles + slots - 1) / slots);
            // The 256 x 512 tile's single accumulator is not handed to the
            // next tile's MMAs until its epilogue has read it all out, which
            // waits on the stores: about 6.5 us less 0.1 us per k-block per
            // wave (the stores of short tiles contend most), and 8 us more
            // for the last epilogue -- fitted on GB300 to 27 shapes timed
            // both ways, K from 512 to 16384.
            const double handover = c.tile_n == 512 ? std::max(0.0, 6.5 - 0.1 * k_blocks) : 0.0;
            cost = waves * (double(k_blocks) * kb_us(c.tile_m, c.tile_n) + handover) +
                   (c.tile_m == 2 * kTileM ? 8.0 : 0.0) + (c.tile_n == 512 ? 8.0 : 0.0);
        }
        if (!best || cost < best_cost) {
            best = &c;
            best_cost = cost;
        }
    }
    if (!best)
        return fail(GEMM_ERR_INVALID_VALUE, "no tile shape matches tile_m=%d tile_n=%d", req_m, req_n);
    const int tm = best->tile_m, bn = best->tile_n;
    int split = K == 0 ? 1 : split_for(tm, bn);
    const int64_t tiles = tiles_of(tm, bn);
    const SmemBudget sb = smem_budget(tm, bn);
    pl->tile_m = tm;
    pl->tile_n = bn;
    pl->tile_k = kTileK;
    pl->stages = sb.stages;
    pl->split_k = split;
    pl->tiles_m = ceil_div(Mx, tm);
    pl->tiles_n = ceil_div(Nx, bn);
    pl->k_blocks = k_blocks;
    pl->units = tiles * split;
    if (pl->units > kInt32Max)
        return fail(GEMM_ERR_INVALID_VALUE, "problem has too many tiles");
    const int64_t ctas_per_unit = tm == 2 * kTileM ? 2 : 1;
    pl->grid = int(std::min<int64_t>(pl->units, slots_of(tm)) * ctas_per_unit);
    pl->group_m = std::min(pl->tiles_m, 8);
    pl->stage_bytes = sb.stage_bytes;
    pl->smem_bytes = sb.smem_bytes;
    // Split-K partials are summed inside the GEMM kernel when every cluster
    // owns exactly one unit (so all splits of a tile run at once) and one
    // reducer's rows of every split fit the idle shared-memory ring (and a
    // TMA box: at most 256 splits).
    const int64_t reducers = int64_t(split) * ctas_per_unit;
    const int64_t rows_per = (tm + reducers - 1) / reducers;
    const int req_r = o ? o->splitk_reduce : 0;
    pl->fused_reduce = split > 1 && req_r != 1 && split <= 256 && pl->units <= slots_of(tm) &&
                       rows_per * bn * 4 * split <= int64_t(sb.stages) * sb.stage_bytes;
    pl->tail_tiles = 0;
    pl->tail_split = 0;
    pl->tail_narrow = 0;
    if (split == 1) {
        const Tail tl = tail_of(tm, bn);
        if (tl.pieces >= 2) {
            pl->tail_tiles = int32_t(tiles % slots_of(tm));
            pl->tail_split = tl.pieces;
            pl->tail_narrow = tl.narrow ? 1 : 0;
            pl->units = tiles - pl->tail_tiles + int64_t(pl->tail_tiles) * tl.pieces;
            pl->grid = int(std::min<int64_t>(pl->units, slots_of(tm)) * ctas_per_unit);
            pl->fused_reduce = tl.narrow ? 0 : 1;
        }
    }
    // Cluster split-K sum (one CTA per tile, every unit a K range summed in
    // the kernel): clusters of CL CTAs hold CL consecutive K ranges of a tile
    // and add them on chip, so only split / CL partials per tile go through
    // the workspace.  The split becomes a multiple of CL that keeps every
    // cluster resident at once (the occupancy API's count), at least 4
    // k-blocks per range.  The idle ring and the epilogue buffers must hold
    // CL receive slots of tile_m / CL rows and the CL - 1 slots a CTA sends,
    // and the slots one reducer's rows of the tile's cluster partials.
    pl->red_cluster = 1;
    // Opt-in: on GB300 the exchange through distributed shared memory costs
    // more than the smaller workspace traffic saves (256 x 256 x 65536:
    // 28.7 us in pairs and 29.8 us in 4-CTA clusters against 27.7 us summed
    // split by split, interleaved on one box), so the planner leaves it off.
    if (pl->fused_reduce && split > 1 && pl->tail_split == 0 && tm == kTileM &&
        (bn == 128 || bn == 256) && (req_c == 2 || req_c == 4)) {
        const int cl = req_c;
        const int64_t cap = cl == 4 ? caps4 : caps2;
        int s2 = 0;
        if (req_s > 0)
            s2 = (split % cl == 0 && tiles * split <= cap * cl) ? split : 0;
        else
            s2 = int(std::min<int64_t>(cap / tiles, k_blocks / (4 * cl))) * cl;
        if (s2 >= cl) {
            const int64_t G = s2 / cl;
            const int64_t rows_own = kTileM / cl;
            const int64_t rp = (rows_own + G - 1) / G;
            const int64_t slot = rows_own * bn * 4;
            const int64_t room = sb.smem_bytes - kSmemSlackAndControl;  // ring + epilogue buffers
            if (G <= 256 && (2 * cl - 1) * slot <= room && rp * G <= kTileM) {
                split = s2;
                pl->split_k = s2;
                pl->units = tiles * s2;
                pl->grid = int(pl->units);
                pl->red_cluster = cl;
            }
        }
    }
    // Split partials: in-kernel sums use a compact [split unit][tile_m][tile_n]
    // workspace (with a cluster sum: [tile * clusters per tile + g]) plus a
    // counter per split tile (per tile and cluster rank) and a 16-byte launch
    // tag; the reduce kernel reads [batch * split][M][ldw].
    const bool ktail = pl->tail_split && !pl->tail_narrow;
    const int64_t split_tiles = ktail ? pl->tail_tiles : (split > 1 ? tiles : 0);
    const int64_t split_units = ktail ? split_tiles * pl->tail_split : split_tiles * split;
    if (split == 1 && !ktail)
        pl->workspace_bytes = 0;
    else if (pl->red_cluster > 1)
        pl->workspace_bytes = split_tiles * (split / pl->red_cluster > 1 ? split / pl->red_cluster : 0) *
                                  tile_elems_of(tm, bn) * 4 +
                              (split_tiles * pl->red_cluster * 4 + 15) / 16 * 16 + 16;
    else if (pl->fused_reduce)
        pl->workspace_bytes = split_units * tile_elems_of(tm, bn) * 4 + (split_tiles * 4 + 15) / 16 * 16 + 16;
    else
        pl->workspace_bytes = batch * int64_t(split) * M * ldw * 4;
    return GEMM_OK;
}

// ------------------------------------------------------------- tensor maps

// Encoding a tensor map is a pure function of its arguments, so each host
// thread keeps its last few maps and hands back the same 128 bytes when a
// call repeats a layout (the usual case: the same operands, or the same
// shapes at the same addresses from a caching allocator).  Nothing about the
// memory behind the address is remembered -- only what the encoder was told.
struct MapKey {
    uint64_t base;
    int64_t cols, rows, mats, ld, stride;
    uint32_t box_cols, box_rows, box_mats;
    int32_t dt, elem, promo, swizzle;
    bool operator==(const MapKey &o) const
    {
        return base == o.base && cols == o.cols && rows == o.rows && mats == o.mats && ld == o.ld &&
               stride == o.stride && box_cols == o.box_cols && box_rows == o.box_rows &&
               box_mats == o.box_mats && dt == o.dt && elem == o.elem && promo == o.promo &&
               swizzle == o.swizzle;
    }
};
struct MapCacheEntry {
    MapKey key;
    alignas(64) CUtensorMap map;
};
constexpr int kMapCacheEntries = 16;
thread_local MapCacheEntry t_map_cache[kMapCacheEntries];
thread_local int t_map_cache_used = 0, t_map_cache_next = 0;

gemm_status_t encode_3d(CUtensorMap *map, CUtensorMapDataType dt, int elem, const void *base,
                        int64_t cols, int64_t rows, int64_t mats, int64_t ld, int64_t stride,
                        uint32_t box_cols, uint32_t box_rows, CUtensorMapL2promotion promo,
                        const char *name, uint32_t box_mats = 1,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    const MapKey key{uint64_t(reinterpret_cast<uintptr_t>(base)), cols, rows, mats, ld, stride,
                     box_cols, box_rows, box_mats, int32_t(dt), elem, int32_t(promo), int32_t(swizzle)};
    for (int i = 0; i < t_map_cache_used; ++i) {
        if (t_map_cache[i].key == key) {
            *map = t_map_cache[i].map;
            return GEMM_OK;
        }
    }
    Driver &d = driver();
    if (!d.loaded)
        return fail(GEMM_ERR_CUDA, "%s", d.error.c_str());
    const cuuint64_t dims[3] = {cuuint64_t(cols), cuuint64_t(rows), cuuint64_t(mats)};
    const cuuint64_t strides[2] = {cuuint64_t(ld) * elem, cuuint64_t(stride) * elem};
    const cuuint32_t box[3] = {box_cols, box_rows, box_mats};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = d.encode_tiled(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GEMM_ERR_INVALID_VALUE, "tensor map for %s rejected (CUresult %d)", name, int(r));
    MapCacheEntry &slot = t_map_cache[t_map_cache_next];
    slot.key = key;
    slot.map = *map;
    t_map_cache_next = (t_map_cache_next + 1) % kMapCacheEntries;
    if (t_map_cache_used < kMapCacheEntries)
        ++t_map_cache_used;
    return GEMM_OK;
}

// ------------------------------------------------------------- the call

int64_t timeout_ns_for(const gemm_options_t *o, const gemm_plan_info_t &pl)
{
    const int64_t base_ms = (o && o->timeout_ms > 0) ? o->timeout_ms : 2000;
    const int64_t kb_per_unit = (pl.k_blocks + pl.split_k - 1) / pl.split_k;
    return base_ms * 1000000ll + kb_per_unit * 10000ll;
}

gemm_status_t run(const Problem &pr, const gemm_options_t *o, cudaStream_t stream);

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// An operand the TMA cannot address (TmaLayout) goes through a packed,
// aligned copy in the pool: A and B are copied in before the GEMM, C is
// computed there and copied out after it -- in a grouped call only the rows
// below each count, so the others stay untouched.  The GEMM between is the
// normal path, so the result is the one the aligned call would give.
gemm_status_t run_repacked(const Problem &pr, const gemm_options_t *o, cudaStream_t stream,
                           DeviceState *ds, const TmaLayout &tl)
{
    const int32_t M = int32_t(pr.M), N = int32_t(pr.N), K = int32_t(pr.K), batch = int32_t(pr.batch);
    const int eb = pr.epi.out_bytes();
    const int64_t lda2 = round_up(pr.K, 8), ldb2 = round_up(pr.N, 8), ldc2 = round_up(pr.N, 16 / eb);
    const int64_t bytesA = tl.a ? 0 : round_up(pr.batch * pr.M * lda2 * 2, 256);
    const int64_t bytesB = tl.b ? 0 : round_up(pr.batch * pr.K * ldb2 * 2, 256);
    const int64_t bytesC = tl.c ? 0 : round_up(pr.batch * pr.M * ldc2 * eb, 256);
    void *scratch = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&scratch, size_t(bytesA + bytesB + bytesC), ds->pool, stream);
    if (e != cudaSuccess)
        return fail_cuda(e, "scratch for repacked operands");
    char *p = static_cast<char *>(scratch);
    const int64_t sA = pr.batch > 1 ? pr.sA : 0, sB = pr.batch > 1 ? pr.sB : 0;
    const int64_t sC = pr.batch > 1 ? pr.sC : 0;
    Problem q = pr;
    gemm_status_t st = GEMM_OK;
    if (!tl.a) {
        uint16_t *A2 = reinterpret_cast<uint16_t *>(p);
        q.A = A2;
        q.lda = lda2;
        q.sA = pr.M * lda2;
        if ((e = launch_pack_f16(pr.A, pr.lda, sA, A2, lda2, q.sA, M, K, batch, ds->sms, stream)) !=
            cudaSuccess)
            st = fail_cuda(e, "repacking A");
    }
    if (st == GEMM_OK && !tl.b) {
        uint16_t *B2 = reinterpret_cast<uint16_t *>(p + bytesA);
        q.B = B2;
        q.ldb = ldb2;
        q.sB = pr.K * ldb2;
        if ((e = launch_pack_f16(pr.B, pr.ldb, sB, B2, ldb2, q.sB, K, N, batch, ds->sms, stream)) !=
            cudaSuccess)
            st = fail_cuda(e, "repacking B");
    }
    if (!tl.c) {
        q.C = p + bytesA + bytesB;
        q.ldc = ldc2;
        q.sC = pr.M * ldc2;
    }
    if (st == GEMM_OK && !tma_layout(q).all())
        st = fail(GEMM_ERR_INVALID_VALUE, "internal: a repacked operand is still misaligned");
    if (st == GEMM_OK)
        st = run(q, o, stream);
    if (st == GEMM_OK && !tl.c) {
        e = eb == 4 ? launch_unpack_f32(static_cast<const float *>(q.C), ldc2, q.sC,
                                        static_cast<float *>(pr.C), pr.ldc, sC, M, N, batch,
                                        pr.group_rows, ds->sms, stream)
                    : launch_unpack_u16(static_cast<const uint16_t *>(q.C), ldc2, q.sC,
                                        static_cast<uint16_t *>(pr.C), pr.ldc, sC, M, N, batch,
                                        pr.group_rows, ds->sms, stream);
        if (e != cudaSuccess)
            st = fail_cuda(e, "copying C out of the repacked layout");
    }
    cudaFreeAsync(scratch, stream);
    return st;
}

gemm_status_t run(const Problem &pr, const gemm_options_t *o, cudaStream_t stream)
{
    bool trivial = false;
    gemm_status_t st = check_host(pr, &trivial);
    if (st != GEMM_OK || trivial)
        return st;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaGetDevice");
    DeviceState *ds = nullptr;
    if ((st = device_state(dev, &ds)) != GEMM_OK)
        return st;

    const int eb = pr.epi.out_bytes();
    const bool use_epi = !pr.epi.identity();
    const int64_t bytesC = span_bytes(pr.batch, pr.sC, pr.M, pr.ldc, pr.N, eb);
    if ((st = check_device_pointer(pr.C, bytesC, dev, "C")) != GEMM_OK)
        return st;
    if (pr.epi.bias &&
        (st = check_device_pointer(pr.epi.bias, span_bytes(pr.batch, pr.epi.bias_stride, 1, pr.N, pr.N, 4),
                                   dev, "bias")) != GEMM_OK)
        return st;
    const int32_t M = int32_t(pr.M), N = int32_t(pr.N), batch = int32_t(pr.batch);
    const int64_t sC = pr.batch > 1 ? pr.sC : int64_t(pr.M) * pr.ldc;
    if (pr.group_rows) {
        if (pr.batch > kMaxGroupsPerLaunch)
            return fail(GEMM_ERR_INVALID_VALUE, "at most %d groups per launch", kMaxGroupsPerLaunch);
        if ((st = check_device_pointer(pr.group_rows, pr.batch * 4, dev, "group_rows")) != GEMM_OK)
            return st;
    }

    if (pr.K == 0) {
        const int64_t total = int64_t(M) * N * batch;
        const int grid = int(std::min<int64_t>((total + 255) / 256, int64_t(ds->sms) * 8));
        if ((e = launch_zero_fill(pr.C, M, N, batch, pr.ldc, sC, pr.group_rows, pr.epi, grid,
                                  stream)) != cudaSuccess)
            return fail_cuda(e, "zero-fill launch");
        return GEMM_OK;
    }

    if ((st = check_device_pointer(pr.A, span_bytes(pr.batch, pr.sA, pr.M, pr.lda, pr.K, 2), dev, "A")) != GEMM_OK)
        return st;
    if ((st = check_device_pointer(pr.B, span_bytes(pr.batch, pr.sB, pr.K, pr.ldb, pr.N, 2), dev, "B")) != GEMM_OK)
        return st;
    const TmaLayout tl = tma_layout(pr);
    if (!tl.all())
        return run_repacked(pr, o, stream, ds, tl);

    // A grouped launch's units are known only on the device, so it takes no
    // split: every unit is a whole tile.
    gemm_options_t og = {};
    if (o)
        og = *o;
    if (pr.group_rows) {
        og.split_k = 1;
        og.split_tail = 2;
    }
    gemm_plan_info_t pl;
    if ((st = make_plan(pr.M, pr.N, pr.K, pr.batch, (o || pr.group_rows) ? &og : nullptr, ds->sms,
                        ds->caps2, ds->caps4, &pl, !pr.group_rows)) != GEMM_OK)
        return st;
    if (ds->smem_optin < pl.smem_bytes)
        return fail(GEMM_ERR_UNSUPPORTED_DEVICE, "device allows %d bytes of shared memory per block, the kernel needs %lld",
                    ds->smem_optin, (long long)pl.smem_bytes);
    const int ti = attr_index(pl.tile_m, pl.tile_n, use_epi, pl.red_cluster, pr.epi.act);
    if (!ds->attrs_set[ti]) {
        if ((e = set_kernel_attributes(pl.tile_m, pl.tile_n, use_epi, pl.red_cluster, pr.epi.act)) != cudaSuccess)
            return fail_cuda(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        ds->attrs_set[ti] = true;
    }

    const int64_t sA = pr.batch > 1 ? pr.sA : int64_t(pr.M) * pr.lda;
    const int64_t sB = pr.batch > 1 ? pr.sB : int64_t(pr.K) * pr.ldb;
    alignas(64) CUtensorMap map_a, map_b, map_out;
    if ((st = encode_3d(&map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, pr.A, pr.K, pr.M, pr.batch,
                        pr.lda, sA, kTileK, kTileM, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "A")) != GEMM_OK)
        return st;
    if ((st = encode_3d(&map_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, pr.B, pr.N, pr.K, pr.batch,
                        pr.ldb, sB, 64, kTileK, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "B")) != GEMM_OK)
        return st;

    KernelParams kp = {};
    kp.M = M;
    kp.N = N;
    kp.K = int32_t(pr.K);
    kp.tiles_m = pl.tiles_m;
    kp.tiles_n = pl.tiles_n;
    kp.k_blocks = pl.k_blocks;
    kp.split_k = pl.split_k;
    kp.batch = batch;
    kp.group_m = pl.group_m;
    kp.inject_stall = (o && o->inject_stall) ? 1 : 0;
    kp.num_units = pl.units;
    kp.timeout_ns = uint64_t(timeout_ns_for(o, pl));
    kp.status = ds->status;
    kp.trace = o ? reinterpret_cast<unsigned long long *>(o->trace) : nullptr;
    kp.group_rows = pr.group_rows;
    kp.groups = pr.group_rows ? batch : 0;
    kp.epi = pr.epi;
    // C's tensor map: f32 boxes of 32 x 32 with the 128-byte swizzle, or
    // 16-bit boxes of 32 x 32 (64-byte rows) with the 64-byte swizzle.  A TMA
    // store writes whole 16-byte granules of a row, so the map ends at the
    // last multiple of 16 bytes and the rest of a row goes by plain stores.
    const int64_t granule = 16 / eb;
    auto encode_out = [&](CUtensorMap *m, int64_t cols) {
        if (eb == 4)
            return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pr.C, cols, pr.M, pr.batch, pr.ldc,
                             sC, 32, 32, CU_TENSOR_MAP_L2_PROMOTION_NONE, "C");
        return encode_3d(m,
                         pr.epi.out_type == kOutBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, pr.C, cols, pr.M, pr.batch, pr.ldc, sC, 32, 32,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, "C", 1, CU_TENSOR_MAP_SWIZZLE_64B);
    };

    kp.n_tma = N;
    kp.tail = 0;
    kp.c_direct = pr.C;
    kp.ldc = pr.ldc;
    kp.stride_c = sC;
    // Asking L2 for a unit's whole K range up front measured slower than the
    // ring's own loads (the burst delays the first k-block), so it is opt-in.
    kp.prefetch_l2 = (o && o->l2_prefetch == 2) ? 1 : 0;
    if (pl.split_k == 1 && !pl.fused_reduce) {
        // TMA stores write whole 16-byte granules: let the map end at the last
        // multiple of 4 columns and write the rest with plain stores, so that
        // C's row padding past N stays untouched.
        if (N % granule) {
            kp.n_tma = int32_t(N & ~(granule - 1));
            kp.tail = 1;
        }
        const int64_t map_cols = kp.n_tma > 0 ? kp.n_tma : pr.N;  // an unused map still needs extent
        if ((st = encode_out(&map_out, map_cols)) != GEMM_OK)
            return st;
        if (pl.tail_narrow) {
            kp.narrow = pl.tail_split;
            kp.dp_units = int64_t(pl.tiles_m) * pl.tiles_n * pr.batch - pl.tail_tiles;
        }
        if ((e = launch_tcgen05_gemm(pl.tile_m, pl.tile_n, use_epi, 1, map_a, map_b, map_out, map_out,
                                     map_out, kp, pl.grid, stream)) != cudaSuccess)
            return fail_cuda(e, "GEMM kernel launch");
        return GEMM_OK;
    }

    if (pl.fused_reduce) {
        // Split partials summed inside the GEMM kernel: one launch.  Split
        // units store their partial tile to the compact workspace
        // [split unit][tile_m][tile_n] (workspace map); each reducer fetches
        // rows_per rows of every split of its tile (reduce map).
        const bool tail = pl.tail_split > 0;
        const int32_t S = tail ? pl.tail_split : pl.split_k;
        const int64_t tiles = int64_t(pl.tiles_m) * pl.tiles_n * pr.batch;
        const int64_t split_tiles = tail ? pl.tail_tiles : tiles;
        const int32_t CL = pl.red_cluster;
        const int32_t G = S / CL;  // partials per tile in the workspace (clusters per tile)
        // With a cluster sum and one cluster per tile nothing goes through the workspace.
        const int64_t split_units = split_tiles * (CL > 1 && G == 1 ? 0 : G);
        const int64_t tile_elems = int64_t(pl.tile_m) * pl.tile_n;
        const int64_t counter_words = split_tiles * CL;
        void *ws = nullptr;
        if ((e = cudaMallocFromPoolAsync(&ws, size_t(pl.workspace_bytes), ds->pool, stream)) != cudaSuccess)
            return fail_cuda(e, "split-K workspace allocation");
        const int64_t cpu = pl.tile_m == 2 * kTileM ? 2 : 1;
        kp.fused = 1;
        kp.split_k = S;
        kp.dp_units = tail ? tiles - split_tiles : 0;
        kp.red_cluster = CL;
        kp.red_groups = G;
        if (CL > 1) {
            kp.reducers = G;
            kp.rows_per = (kTileM / CL + G - 1) / G;
        } else {
            kp.reducers = int32_t(S * cpu);
            kp.rows_per = int32_t((pl.tile_m + kp.reducers - 1) / kp.reducers);
        }
        // CTA pairs with a K-range tail: the split units go first, so that
        // their sums overlap the later tiles (they all fit the first wave).
        kp.split_first = (tail && pl.tile_m == 2 * kTileM) ? 1 : 0;
        kp.n_first = split_units;
        kp.ws = static_cast<const float *>(ws);
        kp.counters = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + split_units * tile_elems * 4);
        kp.counter_words = int32_t(counter_words);
        kp.epoch_tag = reinterpret_cast<unsigned long long *>(
            static_cast<char *>(ws) + split_units * tile_elems * 4 + (counter_words * 4 + 15) / 16 * 16);
        kp.epoch = next_launch_epoch();
        kp.timeout_ns = uint64_t(timeout_ns_for(o, pl));
        alignas(64) CUtensorMap map_ws, map_red;
        // C itself for the whole tiles (and as a valid map to prefetch).
        if (N % granule) {
            kp.n_tma = int32_t(N & ~(granule - 1));
            kp.tail = 1;
        }
        const int64_t map_cols = kp.n_tma > 0 ? kp.n_tma : pr.N;
        st = encode_out(&map_out, map_cols);
        // (A cluster sum with one cluster per tile uses neither workspace
        // map; they still need a valid extent to be prefetched.)
        const int64_t ws_mats = std::max<int64_t>(split_units, 1);
        if (st == GEMM_OK)
            st = encode_3d(&map_ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, pl.tile_n, pl.tile_m,
                           ws_mats, pl.tile_n, tile_elems, 32, 32,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, "split-K workspace");
        if (st == GEMM_OK)
            st = encode_3d(&map_red, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, pl.tile_n, pl.tile_m,
                           ws_mats, pl.tile_n, tile_elems, uint32_t(pl.tile_n),
                           uint32_t(kp.rows_per), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           "split-K workspace (reduce)", uint32_t(G), CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st == GEMM_OK &&
            (e = launch_tcgen05_gemm(pl.tile_m, pl.tile_n, use_epi, CL, map_a, map_b, map_out, map_ws,
                                     map_red, kp, pl.grid, stream)) != cudaSuccess)
            st = fail_cuda(e, "GEMM kernel launch");
        cudaFreeAsync(ws, stream);
        return st;
    }

    // Split-K: partials W[b*S + s] (M x ldw f32 each), then the fixed-order sum.
    const int64_t ldw = (pr.N + 3) / 4 * 4;
    void *ws = nullptr;
    if ((e = cudaMallocFromPoolAsync(&ws, size_t(pl.workspace_bytes), ds->pool, stream)) != cudaSuccess)
        return fail_cuda(e, "split-K workspace allocation");
    st = encode_3d(&map_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, pr.N, pr.M,
                   pr.batch * pl.split_k, ldw, int64_t(pr.M) * ldw, 32, 32,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, "split-K workspace");
    // The GEMM writes raw partials (the plain kernel); the reduce applies
    // the epilogue to the sums.
    kp.epi = Epilogue{};
    if (st == GEMM_OK && !ds->attrs_set[attr_index(pl.tile_m, pl.tile_n, false, 1, kActNone)]) {
        if ((e = set_kernel_attributes(pl.tile_m, pl.tile_n, false)) != cudaSuccess)
            st = fail_cuda(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        else
            ds->attrs_set[attr_index(pl.tile_m, pl.tile_n, false, 1, kActNone)] = true;
    }
    if (st == GEMM_OK) {
        if ((e = launch_tcgen05_gemm(pl.tile_m, pl.tile_n, false, 1, map_a, map_b, map_out, map_out,
                                     map_out, kp, pl.grid, stream)) != cudaSuccess)
            st = fail_cuda(e, "GEMM kernel launch");
    }
    if (st == GEMM_OK) {
        const int64_t threads = int64_t(M) * ((N + 3) / 4) * batch;
        const int grid = int(std::min<int64_t>((threads + 255) / 256, int64_t(ds->sms) * 8));
        if ((e = launch_splitk_reduce(static_cast<const float *>(ws), pr.C, M, N, pl.split_k, batch,
                                      ldw, pr.ldc, sC, pr.epi, grid, stream)) != cudaSuccess)
            st = fail_cuda(e, "split-K reduce launch");
    }
    cudaFreeAsync(ws, stream);
    return st;
}

}  // namespace
}  // namespace tsm

using namespace tsm;

extern "C" {

gemm_status_t gemm_f16_f32acc(const uint16_t *A, const uint16_t *B, float *C, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, int64_t ldc, gemm_stream_t stream)
{
    g_last_error.clear();
    Problem pr{A, B, C, M, N, K, lda, ldb, ldc, 0, 0, 0, 1};
    return run(pr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16_f32acc_batched(const uint16_t *A, const uint16_t *B, float *C, int64_t M,
                                      int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                      int64_t strideA, int64_t strideB, int64_t strideC,
                                      int64_t batch, gemm_stream_t stream)
{
    g_last_error.clear();
    Problem pr{A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, batch};
    return run(pr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16_f32acc_opts(const uint16_t *A, const uint16_t *B, float *C, int64_t M,
                                   int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                   int64_t strideA, int64_t strideB, int64_t strideC, int64_t batch,
                                   const gemm_options_t *opts, gemm_stream_t stream)
{
    g_last_error.clear();
    Problem pr{A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, batch};
    return run(pr, opts, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace tsm {
namespace {

// A row reduction (rowsum_kernels.cu): the launch shape from (R, C) and the
// layout alone, so that the summation order -- and the result -- is the same
// on every call.  16-byte vector loads when the rows are contiguous and
// 16-byte aligned; each lane takes at least 32 chunks (or elements) of a
// row where the row is long enough; rows too few to fill the GPU are cut
// into segments whose partial sums a second kernel adds in order.
gemm_status_t row_reduce(const void *X, int elem, int64_t R, int64_t C, int64_t row_stride,
                         int64_t col_stride, const uint16_t *xv, int64_t incx, float *out,
                         cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaGetDevice");
    DeviceState *ds = nullptr;
    gemm_status_t st = device_state(dev, &ds);
    if (st != GEMM_OK)
        return st;
    const int eb = elem == kOutF32 ? 4 : 2;
    const int64_t V = 16 / eb;
    const int64_t span = C > 0 ? ((R - 1) * row_stride + (C - 1) * col_stride + 1) * eb : 0;
    if (C > 0 && (st = check_device_pointer(X, span, dev, xv ? "A" : "X")) != GEMM_OK)
        return st;
    if (xv && C > 0 && (st = check_device_pointer(xv, ((C - 1) * incx + 1) * 2, dev, "x")) != GEMM_OK)
        return st;
    if ((st = check_device_pointer(out, R * 4, dev, xv ? "y" : "out")) != GEMM_OK)
        return st;

    bool vec = C >= V && col_stride == 1 && !(reinterpret_cast<uintptr_t>(X) & 15u) &&
               (R == 1 || (row_stride * eb) % 16 == 0);
    if (xv)
        vec = vec && incx == 1 && !(reinterpret_cast<uintptr_t>(xv) & 15u);
    const int64_t units = vec ? C / V : C;  // per row
    int tpr = 1;
    while (tpr < 32 && int64_t(tpr) * 32 <= units)
        tpr *= 2;
    const int64_t per_block = 8 * (32 / tpr);  // workers in a block of 8 warps
    const int64_t resident = int64_t(ds->sms) * row_reduce_blocks_per_sm(elem, vec, xv != nullptr);
    const int64_t max_workers = resident * per_block;  // workers that run at once
    int64_t segs = 1;
    if (R < max_workers && C > 0)
        // Rounded down: R x segs items at most the workers that fit at once
        // (one full pass; rounding up made two half-empty ones, measured 1.9x
        // slower at 1024 x 131072 f32).
        segs = std::max<int64_t>(1, std::min<int64_t>(max_workers / R,
                                                      std::min<int64_t>(units / (16 * tpr), 65536)));
    int64_t seg = C > 0 ? (C + segs - 1) / segs : 0;
    if (vec)
        seg = (seg + V - 1) / V * V;
    if (C > 0)
        segs = (C + seg - 1) / seg;
    // As many workers as give every one the same number of items: the items
    // in `rounds` even passes, not a last pass half empty.
    const int64_t items = R * segs;
    const int64_t rounds = (items + max_workers - 1) / max_workers;
    const int64_t want = (items + rounds - 1) / rounds;
    const int grid = int(std::max<int64_t>(1, (want + per_block - 1) / per_block));

    RowReduceParams p = {};
    p.X = X;
    p.row_stride = row_stride;
    p.col_stride = col_stride;
    p.xv = xv;
    p.incx = incx;
    p.out = out;
    p.R = R;
    p.C = C;
    p.seg = std::max<int64_t>(seg, 1);
    p.segs = int32_t(segs);
    p.tpr = tpr;
    void *ws = nullptr;
    if (segs > 1) {
        if ((e = cudaMallocFromPoolAsync(&ws, size_t(R * segs * 4), ds->pool, stream)) != cudaSuccess)
            return fail_cuda(e, "row-reduction partials");
        p.partial = static_cast<float *>(ws);
    }
    if ((e = launch_row_reduce(p, elem, vec, xv != nullptr, grid, stream)) != cudaSuccess)
        st = fail_cuda(e, "row-reduction launch");
    if (st == GEMM_OK && segs > 1 &&
        (e = launch_row_partials(p.partial, out, R, int32_t(segs),
                                 int(std::min<int64_t>((R + 7) / 8, int64_t(ds->sms) * 8)), stream)) !=
            cudaSuccess)
        st = fail_cuda(e, "row-partials launch");
    if (ws)
        cudaFreeAsync(ws, stream);
    return st;
}

}  // namespace
}  // namespace tsm

extern "C" {

gemm_status_t rowsum_f32acc(const void *X, int32_t elem_type, float *out, int64_t R, int64_t C,
                            int64_t row_stride, int64_t col_stride, gemm_stream_t stream)
{
    g_last_error.clear();
    if (elem_type != GEMM_OUT_F32 && elem_type != GEMM_OUT_F16 && elem_type != GEMM_OUT_BF16)
        return fail(GEMM_ERR_INVALID_VALUE, "unknown element type %d", elem_type);
    if (R < 0 || C < 0 || R > (int64_t(1) << 40) || C > (int64_t(1) << 40))
        return fail(GEMM_ERR_INVALID_VALUE, "bad size: R=%lld C=%lld", (long long)R, (long long)C);
    if (R == 0)
        return GEMM_OK;
    if (!out || (C > 0 && !X))
        return fail(GEMM_ERR_INVALID_VALUE, "X or out is NULL");
    if (row_stride < 0 || (C > 1 && col_stride < 1))
        return fail(GEMM_ERR_INVALID_VALUE, "row_stride must be >= 0 and col_stride >= 1");
    const int eb = elem_type == GEMM_OUT_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(X) & uintptr_t(eb - 1)) || (reinterpret_cast<uintptr_t>(out) & 3u))
        return fail(GEMM_ERR_MISALIGNED, "X and out must sit at their elements' natural alignment");
    const int64_t span = C > 0 ? ((R - 1) * row_stride + (C - 1) * col_stride + 1) * eb : 0;
    if (overlaps(out, R * 4, X, span))
        return fail(GEMM_ERR_ALIAS, "out overlaps X");
    return row_reduce(X, elem_type, R, C, row_stride, C > 1 ? col_stride : 1, nullptr, 0, out,
                      reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemv_f16_f32acc(const uint16_t *A, const uint16_t *x, float *y, int64_t M, int64_t K,
                              int64_t lda, int64_t incx, gemm_stream_t stream)
{
    g_last_error.clear();
    if (M < 0 || K < 0 || M > (int64_t(1) << 40) || K > (int64_t(1) << 40))
        return fail(GEMM_ERR_INVALID_VALUE, "bad size: M=%lld K=%lld", (long long)M, (long long)K);
    if (M == 0)
        return GEMM_OK;
    if (!y || (K > 0 && (!A || !x)))
        return fail(GEMM_ERR_INVALID_VALUE, "A, x or y is NULL");
    if (lda < K || (K > 1 && incx < 1))
        return fail(GEMM_ERR_INVALID_VALUE, "lda must be >= K and incx >= 1");
    if ((reinterpret_cast<uintptr_t>(A) & 1u) || (reinterpret_cast<uintptr_t>(x) & 1u) ||
        (reinterpret_cast<uintptr_t>(y) & 3u))
        return fail(GEMM_ERR_MISALIGNED, "A and x must be 2-byte and y 4-byte aligned");
    const int64_t spanA = K > 0 ? ((M - 1) * lda + K) * 2 : 0;
    const int64_t spanx = K > 0 ? ((K - 1) * incx + 1) * 2 : 0;
    if (overlaps(y, M * 4, A, spanA) || overlaps(y, M * 4, x, spanx))
        return fail(GEMM_ERR_ALIAS, "y overlaps A or x");
    return row_reduce(A, GEMM_OUT_F16, M, K, lda, 1, x, K > 1 ? incx : 1, y,
                      reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace tsm {
namespace {

// The public epilogue description, checked, as the kernels' Epilogue.
gemm_status_t epilogue_of(const gemm_epilogue_t *e, Epilogue *out)
{
    *out = Epilogue{};
    if (!e)
        return GEMM_OK;
    if (e->activation < GEMM_ACT_NONE || e->activation > GEMM_ACT_SILU)
        return fail(GEMM_ERR_INVALID_VALUE, "unknown activation %d", e->activation);
    if (e->out_type < GEMM_OUT_F32 || e->out_type > GEMM_OUT_BF16)
        return fail(GEMM_ERR_INVALID_VALUE, "unknown output type %d", e->out_type);
    out->alpha = e->alpha;
    out->bias = e->bias;
    out->bias_stride = e->bias_stride;
    out->act = e->activation;
    out->slope = e->slope;
    out->out_type = e->out_type;
    return GEMM_OK;
}

// Grouped calls: launches of at most kMaxGroupsPerLaunch groups, in stream order.
gemm_status_t grouped(const uint16_t *A, const uint16_t *B, void *C, const int32_t *group_rows,
                      int64_t groups, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                      int64_t ldc, int64_t strideA, int64_t strideB, int64_t strideC,
                      const Epilogue &epi, const gemm_options_t *opts, cudaStream_t stream)
{
    if (groups < 0)
        return fail(GEMM_ERR_INVALID_VALUE, "negative number of groups: %lld", (long long)groups);
    if (groups > 0 && !group_rows)
        return fail(GEMM_ERR_INVALID_VALUE, "group_rows is NULL");
    if (reinterpret_cast<uintptr_t>(group_rows) & 3u)
        return fail(GEMM_ERR_MISALIGNED, "group_rows must be 4-byte aligned");
    for (int64_t g0 = 0; g0 < groups; g0 += kMaxGroupsPerLaunch) {
        const int64_t n = std::min<int64_t>(kMaxGroupsPerLaunch, groups - g0);
        Problem pr{A ? A + g0 * strideA : A, B ? B + g0 * strideB : B,
                   C ? static_cast<char *>(C) + g0 * strideC * epi.out_bytes() : C,
                   M, N, K, lda, ldb, ldc, strideA, strideB, strideC, n};
        pr.group_rows = group_rows + g0;
        pr.epi = epi;
        if (epi.bias)
            pr.epi.bias = epi.bias + g0 * epi.bias_stride;
        const gemm_status_t st = run(pr, opts, stream);
        if (st != GEMM_OK)
            return st;
    }
    return GEMM_OK;
}

// The planner on the host: the SM count and cluster capacities of the
// current device when num_sms <= 0, else the GB300 estimate for num_sms SMs.
gemm_status_t host_plan(int64_t M, int64_t N, int64_t K, int64_t batch, const gemm_options_t *opts,
                        int32_t num_sms, gemm_plan_info_t *plan, bool wide)
{
    if (!plan)
        return fail(GEMM_ERR_INVALID_VALUE, "plan is NULL");
    if (M < 0 || N < 0 || K < 0 || batch < 0 || M > kInt32Max || N > kInt32Max || K > kInt32Max ||
        batch > kInt32Max)
        return fail(GEMM_ERR_INVALID_VALUE, "sizes must be in [0, 2^31)");
    int sms = num_sms;
    if (sms <= 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return fail_cuda(e, "cudaGetDevice");
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
    }
    int caps2 = estimated_cluster_capacity(sms, 2), caps4 = estimated_cluster_capacity(sms, 4);
    if (num_sms <= 0) {
        int dev = 0;
        DeviceState *ds = nullptr;
        if (cudaGetDevice(&dev) == cudaSuccess && device_state(dev, &ds) == GEMM_OK) {
            caps2 = ds->caps2;
            caps4 = ds->caps4;
        }
        g_last_error.clear();
    }
    return make_plan(M, N, K, std::max<int64_t>(batch, 1), opts, sms, caps2, caps4, plan, wide);
}

}  // namespace
}  // namespace tsm

extern "C" {

gemm_status_t gemm_f16_f32acc_grouped_opts(const uint16_t *A, const uint16_t *B, float *C,
                                           const int32_t *group_rows, int64_t groups, int64_t M,
                                           int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                           int64_t strideA, int64_t strideB, int64_t strideC,
                                           const gemm_options_t *opts, gemm_stream_t stream)
{
    g_last_error.clear();
    return grouped(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc, strideA, strideB, strideC,
                   Epilogue{}, opts, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16_f32acc_grouped(const uint16_t *A, const uint16_t *B, float *C,
                                      const int32_t *group_rows, int64_t groups, int64_t M, int64_t N,
                                      int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t strideA,
                                      int64_t strideB, int64_t strideC, gemm_stream_t stream)
{
    return gemm_f16_f32acc_grouped_opts(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc, strideA,
                                        strideB, strideC, nullptr, stream);
}

gemm_status_t gemm_f16_fused(const uint16_t *A, const uint16_t *B, void *C, int64_t M, int64_t N,
                             int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t strideA,
                             int64_t strideB, int64_t strideC, int64_t batch,
                             const gemm_epilogue_t *epi, const gemm_options_t *opts,
                             gemm_stream_t stream)
{
    g_last_error.clear();
    Problem pr{A, B, C, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, batch};
    const gemm_status_t st = epilogue_of(epi, &pr.epi);
    if (st != GEMM_OK)
        return st;
    return run(pr, opts, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16_grouped_fused(const uint16_t *A, const uint16_t *B, void *C,
                                     const int32_t *group_rows, int64_t groups, int64_t M, int64_t N,
                                     int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                     int64_t strideA, int64_t strideB, int64_t strideC,
                                     const gemm_epilogue_t *epi, const gemm_options_t *opts,
                                     gemm_stream_t stream)
{
    g_last_error.clear();
    Epilogue e;
    const gemm_status_t st = epilogue_of(epi, &e);
    if (st != GEMM_OK)
        return st;
    return grouped(A, B, C, group_rows, groups, M, N, K, lda, ldb, ldc, strideA, strideB, strideC, e,
                   opts, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, int64_t batch, const gemm_options_t *opts,
                        int32_t num_sms, gemm_plan_info_t *plan)
{
    g_last_error.clear();
    return tsm::host_plan(M, N, K, batch, opts, num_sms, plan, true);
}

gemm_status_t gemm_plan_grouped(int64_t M, int64_t N, int64_t K, int64_t groups,
                                const gemm_options_t *opts, int32_t num_sms, gemm_plan_info_t *plan)
{
    g_last_error.clear();
    // What a grouped launch plans with: whole tiles (its units are known
    // only on the device), and the 512-column tile only when asked for
    // (measured 1 % slower on 8 experts of 4096 x 14336, K 4096, whose
    // routed rows leave the planner's full-M count of tiles too high).
    gemm_options_t og = {};
    if (opts)
        og = *opts;
    og.split_k = 1;
    og.split_tail = 2;
    return tsm::host_plan(M, N, K, std::min<int64_t>(std::max<int64_t>(groups, 1), kMaxGroupsPerLaunch),
                          &og, num_sms, plan, false);
}

gemm_status_t gemm_get_device_status(gemm_stream_t stream)
{
    g_last_error.clear();
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaStreamSynchronize");
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess)
        return fail_cuda(e, "cudaGetDevice");
    DeviceState *ds = nullptr;
    gemm_status_t st = device_state(dev, &ds);
    if (st != GEMM_OK)
        return st;
    uint32_t word = 0;
    if ((e = cudaMemcpy(&word, ds->status, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail_cuda(e, "reading the status word");
    if (word == 0)
        return GEMM_OK;
    const uint32_t zero = 0;
    cudaMemcpy(ds->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (word == kStatusGroupRows)
        return fail(GEMM_ERR_INVALID_VALUE,
                    "a grouped call had a row count outside [0, M]; it was clamped to that range");
    return fail(GEMM_ERR_DEVICE_TIMEOUT,
                "a bounded device-side wait ran out (roles: %s%s%s%s%s); the output of that call is incomplete",
                (word & kStatusProducer) ? "producer " : "", (word & kStatusMma) ? "mma " : "",
                (word & kStatusEpilogue) ? "epilogue " : "", (word & kStatusDrain) ? "drain " : "",
                (word & kStatusReduce) ? "split-K-reduce" : "");
}

const char *gemm_last_error_string(void) { return g_last_error.c_str(); }

const char *gemm_status_string(gemm_status_t s)
{
    switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE";
    case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED";
    case GEMM_ERR_ALIAS: return "GEMM_ERR_ALIAS";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT";
    }
    return "GEMM_ERR_UNKNOWN";
}

int32_t gemm_version(void) { return 100; }

}  // extern "C"

// ------------------------------------------------------------- no-allocation entry point
//
// Some callers cannot allocate device memory at call time: code running
// inside a CUDA stream capture that must not add allocation nodes, an
// allocator or memory-accounting layer that may not re-enter itself, or an
// embedded host that reserved every byte of the GPU up front.  For them the
// split-K path can take its partial sums from a fixed array that lives in
// this file instead of the stream-ordered pool.  The array is a file-scope
// __device__ object: every GPU that loads the library holds it until the
// process exits.

namespace tsm {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB of f32 partials

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

struct NoAllocDevice {
    bool ready = false;
    void *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int sms = 0;
    int smem_optin = 0;
    uint32_t *status = nullptr;
    bool attrs_set[5] = {false, false, false, false, false};
};

NoAllocDevice g_noalloc_devices[kMaxDevices];
std::mutex g_noalloc_mutex;

// Once per device, with that device current: resolve the array's device
// address (the host-side name is only a stand-in), the SM count and the
// status word.  None of this allocates.
gemm_status_t noalloc_setup(int dev, NoAllocDevice **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GEMM_ERR_INVALID_VALUE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice &d = g_noalloc_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        cudaError_t e;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute(compute capability)");
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(GEMM_ERR_UNSUPPORTED_DEVICE,
                        "device %d has compute capability %d.%d; this library is built for 10.3 only",
                        dev, major, minor);
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if ((e = cudaGetSymbolAddress(&d.scratch, g_noalloc_scratch)) != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(static split-K scratch)");
        if ((e = device_status_word(&d.status)) != cudaSuccess)
            return fail_cuda(e, "cudaGetSymbolAddress(status word)");
        d.ready = true;
    }
    *out = &d;
    return GEMM_OK;
}

// The kernel's shared-memory limit, set once per device and tile shape
// (under the same lock as the set-up, so two host threads making their first
// calls at once do not both write the flag).
gemm_status_t noalloc_kernel_attributes(NoAllocDevice *nd, int tile_m, int tile_n)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const int ti = config_index(tile_m, tile_n);
    if (!nd->attrs_set[ti]) {
        const cudaError_t e = set_kernel_attributes(tile_m, tile_n, false);
        if (e != cudaSuccess)
            return fail_cuda(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        nd->attrs_set[ti] = true;
    }
    return GEMM_OK;
}

}  // namespace
}  // namespace tsm

extern "C" gemm_status_t gemm_f16_f32acc_splitk_noalloc(const uint16_t *A, const uint16_t *B,
                                                        float *C, int64_t M, int64_t N, int64_t K,
                                                        int64_t lda, int64_t ldb, int64_t ldc,
                                                        int32_t split_k, gemm_stream_t stream_)
{
    using namespace tsm;
    g_last_error.clear();
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    Problem pr{A, B, C, M, N, K, lda, ldb, ldc, 0, 0, 0, 1};
    bool trivial = false;
    gemm_status_t st = check_host(pr, &trivial);
    if (st != GEMM_OK || trivial)
        return st;
    if (split_k < 0)
        return fail(GEMM_ERR_INVALID_VALUE, "split_k must be >= 0");
    if (K == 0)
        return fail(GEMM_ERR_INVALID_VALUE, "K == 0 is not served by the no-allocation entry point");
    if (!tma_layout(pr).all())
        return fail(GEMM_ERR_MISALIGNED,
                    "the no-allocation entry point cannot repack: A and B need 16-byte aligned bases "
                    "and lda, ldb multiples of 8 elements, C a 16-byte aligned base and ldc a "
                    "multiple of 4");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaGetDevice");
    NoAllocDevice *nd = nullptr;
    if ((st = noalloc_setup(dev, &nd)) != GEMM_OK)
        return st;
    if ((st = check_device_pointer(C, span_bytes(1, 0, M, ldc, N, 4), dev, "C")) != GEMM_OK)
        return st;
    if ((st = check_device_pointer(A, span_bytes(1, 0, M, lda, K, 2), dev, "A")) != GEMM_OK)
        return st;
    if ((st = check_device_pointer(B, span_bytes(1, 0, K, ldb, N, 2), dev, "B")) != GEMM_OK)
        return st;

    gemm_options_t o = {};
    o.split_k = split_k;
    o.splitk_reduce = 1;  // partials in the scratch, summed by the separate reduce kernel
    gemm_plan_info_t pl;
    if ((st = make_plan(M, N, K, 1, &o, nd->sms, 0, 0, &pl, false)) != GEMM_OK)
        return st;
    if (split_k == 0 && uint64_t(pl.workspace_bytes) > kNoAllocScratchBytes) {
        // The planner's split does not fit: take the largest split that does.
        const int64_t per_split = M * ((N + 3) / 4 * 4) * 4;
        o.split_k = int32_t(std::max<int64_t>(1, int64_t(kNoAllocScratchBytes) / per_split));
        if ((st = make_plan(M, N, K, 1, &o, nd->sms, 0, 0, &pl, false)) != GEMM_OK)
            return st;
    }
    if (uint64_t(pl.workspace_bytes) > kNoAllocScratchBytes)
        return fail(GEMM_ERR_INVALID_VALUE,
                    "split-K partials need %lld bytes (S=%d x %lld x %lld f32); the static scratch "
                    "holds %zu bytes -- use a smaller split_k or gemm_f16_f32acc",
                    (long long)pl.workspace_bytes, pl.split_k, (long long)M, (long long)((N + 3) / 4 * 4),
                    kNoAllocScratchBytes);
    if (nd->smem_optin < pl.smem_bytes)
        return fail(GEMM_ERR_UNSUPPORTED_DEVICE, "device allows %d bytes of shared memory per block, the kernel needs %lld",
                    nd->smem_optin, (long long)pl.smem_bytes);
    if ((st = noalloc_kernel_attributes(nd, pl.tile_m, pl.tile_n)) != GEMM_OK)
        return st;

    alignas(64) CUtensorMap map_a, map_b, map_out;
    if ((st = encode_3d(&map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, A, K, M, 1, lda, M * lda, kTileK,
                        kTileM, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "A")) != GEMM_OK)
        return st;
    if ((st = encode_3d(&map_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, B, N, K, 1, ldb, K * ldb, 64,
                        kTileK, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "B")) != GEMM_OK)
        return st;

    KernelParams kp = {};
    kp.M = int32_t(M);
    kp.N = int32_t(N);
    kp.K = int32_t(K);
    kp.tiles_m = pl.tiles_m;
    kp.tiles_n = pl.tiles_n;
    kp.k_blocks = pl.k_blocks;
    kp.split_k = pl.split_k;
    kp.batch = 1;
    kp.group_m = pl.group_m;
    kp.inject_stall = 0;
    kp.num_units = pl.units;
    kp.timeout_ns = uint64_t(timeout_ns_for(nullptr, pl));
    kp.status = nd->status;
    kp.n_tma = int32_t(N);
    kp.tail = 0;
    kp.c_direct = C;
    kp.ldc = ldc;
    kp.stride_c = M * ldc;

    if (pl.split_k == 1) {
        // No partials to keep: the ordinary single-pass kernel, which needs no scratch.
        if (N % 4) {
            kp.n_tma = int32_t(N) & ~3;
            kp.tail = 1;
        }
        const int64_t map_cols = kp.n_tma > 0 ? kp.n_tma : N;
        if ((st = encode_3d(&map_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, map_cols, M, 1, ldc,
                            M * ldc, 32, 32, CU_TENSOR_MAP_L2_PROMOTION_NONE, "C")) != GEMM_OK)
            return st;
        if (pl.tail_narrow) {
            kp.narrow = pl.tail_split;
            kp.dp_units = int64_t(pl.tiles_m) * pl.tiles_n - pl.tail_tiles;
        }
        if ((e = launch_tcgen05_gemm(pl.tile_m, pl.tile_n, false, 1, map_a, map_b, map_out, map_out,
                                     map_out, kp, pl.grid, stream)) != cudaSuccess)
            return fail_cuda(e, "GEMM kernel launch");
        return GEMM_OK;
    }

    // Every (split, row < M, column < N) partial is written before the reduce
    // reads it, so nothing in the scratch has to start at zero.
    const int64_t ldw = (N + 3) / 4 * 4;
    if ((st = encode_3d(&map_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, nd->scratch, N, M, pl.split_k,
                        ldw, M * ldw, 32, 32, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        "static split-K scratch")) != GEMM_OK)
        return st;
    if ((e = launch_tcgen05_gemm(pl.tile_m, pl.tile_n, false, 1, map_a, map_b, map_out, map_out,
                                 map_out, kp, pl.grid, stream)) != cudaSuccess)
        return fail_cuda(e, "GEMM kernel launch");
    const int64_t threads = M * ((N + 3) / 4);
    const int grid = int(std::min<int64_t>((threads + 255) / 256, int64_t(nd->sms) * 8));
    if ((e = launch_splitk_reduce(static_cast<const float *>(nd->scratch), C, int32_t(M), int32_t(N),
                                  pl.split_k, 1, ldw, ldc, M * ldc, Epilogue{}, grid, stream)) != cudaSuccess)
        return fail_cuda(e, "split-K reduce launch");
    return GEMM_OK;
}
