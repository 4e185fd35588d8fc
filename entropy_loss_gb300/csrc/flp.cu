// flp.cu - host side of the C ABI declared in include/flp.h: argument
// validation, workspace layout, schedule choice, TMA tensor maps and launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "flp.h"
#include "bwd.cuh"
#include "kernels.cuh"
#include "loss.cuh"

using namespace flp;

namespace {

thread_local std::string g_msg;

// Named host range for profilers (NVTX; a no-op unless a tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kMaxPhaseEvents = 10;
thread_local void* g_events[kMaxPhaseEvents] = {};
thread_local int g_num_events = 0;

// Records the caller's instrumentation event `idx` (if any) on stream s.
void mark(int idx, cudaStream_t s) {
    if (idx < g_num_events && g_events[idx])
        cudaEventRecord(static_cast<cudaEvent_t>(g_events[idx]), s);
}

flp_status fail(flp_status st, const char* what) {
    g_msg = what;
    return st;
}

flp_status cuda_fail(cudaError_t e, const char* where) {
    char buf[256];
    snprintf(buf, sizeof buf, "%s: %s", where, cudaGetErrorString(e));
    g_msg = buf;
    return FLP_ERR_CUDA;
}

#define FLP_CUDA(call)                                         \
    do {                                                       \
        cudaError_t e_ = (call);                               \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);    \
    } while (0)

constexpr int kMaxDevices = 64;
constexpr size_t kHeaderBytes = 1024;      // error word, ticket counter; keeps regions 1 KiB aligned
constexpr size_t kTicketOffset = 8;        // 64-bit tile ticket counter of the backward contractions
constexpr int64_t kDefaultChunkRows = 8192;
constexpr unsigned long long kWaitLimitNs = 10ull * 1000 * 1000 * 1000;  // 10 s per wait

struct DevInfo {
    bool init = false;
    cudaError_t err = cudaSuccess;
    int sm_count = 0;
    int major = 0, minor = 0;
    bool attrs_set = false;
    int pairs = 0;  // CTA pairs that can be resident at once (persistent grid size / 2)
};
DevInfo g_dev[kMaxDevices];
std::mutex g_mu;

flp_status device_info(DevInfo** out, int* dev_out) {
    int dev = 0;
    FLP_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev];
    if (!d.init) {
        cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        d.init = true;
    }
    *out = &d;
    if (dev_out) *dev_out = dev;
    return FLP_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

flp_status get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDriverEntryPointByVersion");
        if (q != cudaDriverEntryPointSuccess || !p)
            return fail(FLP_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    *fn = g_encode;
    return FLP_OK;
}

// 2-D tiled tensor map, 128-byte swizzle, zero fill outside the tensor.
flp_status tmap_2d(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t inner,
                   uint64_t outer, uint64_t row_pitch_bytes, uint32_t box_inner,
                   uint32_t box_outer, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    flp_status st = get_encode(&enc);
    if (st != FLP_OK) return st;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) dims %llu x %llu pitch %llu",
                 static_cast<int>(r), (unsigned long long)inner, (unsigned long long)outer,
                 (unsigned long long)row_pitch_bytes);
        g_msg = buf;
        return FLP_ERR_CUDA;
    }
    return FLP_OK;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------ forward plan

struct FwdPlan {
    int Mt, Vt, S, tps, GM, units, grid;
    size_t off_m, off_s, off_t, off_zy, bytes;
};

// Chooses the V-split: units are (256-row pair tile, run of tps 512-column
// tiles); a static round-robin over the persistent CTA pairs finishes after
// ceil(units / pairs) * tps tiles.  Each extra split adds M * 48 bytes of
// partial traffic (two halves of m, sigma, tau and their reads), charged in
// tile-times so that near-ties favour fewer splits.  Only plans whose
// workspace fits max_bytes are considered (the allocation-free forward's
// fixed scratch); when none does, the one-split plan is returned and the
// caller sees its size.
FwdPlan plan_forward(int64_t M, int64_t H, int64_t V, int compute_entropy, int pairs,
                     size_t max_bytes = SIZE_MAX) {
    FwdPlan f{};
    pairs = std::max(1, pairs);
    f.Mt = static_cast<int>(cdiv(M, PM));
    f.Vt = static_cast<int>(cdiv(V, 2 * BN));  // 512-column tiles
    const double tile_s = 2.0 * PM * 2 * BN * static_cast<double>(H) / 2.4e13;  // ~bf16 rate of a pair
    const double split_cost = (static_cast<double>(M) * 48.0 / 6.0e12) / tile_s;
    // workspace of a plan with S splits: header | m, sigma (, tau) [2 S][M] | z_y [M]
    auto bytes_for = [&](int S) {
        const size_t part = align_up(static_cast<size_t>(2 * S) * M * sizeof(float), 1024);  // 2 halves per split
        return kHeaderBytes + part * (compute_entropy ? 3 : 2) +
               align_up(static_cast<size_t>(M) * sizeof(float), 1024);
    };
    double best = 1e300;
    int best_tps = f.Vt;
    for (int tps = 1; tps <= f.Vt; ++tps) {
        const int S = static_cast<int>(cdiv(f.Vt, tps));
        if (tps > 1 && cdiv(f.Vt, tps - 1) == S) continue;  // same split count, shorter runs win
        if (bytes_for(S) > max_bytes) continue;
        const double units = static_cast<double>(f.Mt) * S;
        const double waves = std::ceil(units / pairs);
        const double cost = waves * tps + S * split_cost;
        if (cost < best - 1e-9) {
            best = cost;
            best_tps = tps;
        }
    }
    f.tps = best_tps;
    f.S = static_cast<int>(cdiv(f.Vt, f.tps));
    // group of pair M-tiles whose X rows stay resident in L2 (about 40 MB of X)
    const int64_t gm = std::max<int64_t>(4, 40ll * 1000 * 1000 / (PM * 2 * std::max<int64_t>(H, 1)));
    f.GM = static_cast<int>(std::min<int64_t>(f.Mt, gm));
    if (f.GM < 1) f.GM = 1;
    f.units = f.Mt * f.S;
    f.grid = 2 * std::min(f.units, pairs);
    const size_t part = align_up(static_cast<size_t>(2 * f.S) * M * sizeof(float), 1024);  // 2 halves per split
    f.off_m = kHeaderBytes;
    f.off_s = f.off_m + part;
    f.off_t = f.off_s + part;
    f.off_zy = f.off_t + (compute_entropy ? part : 0);
    f.bytes = f.off_zy + align_up(static_cast<size_t>(M) * sizeof(float), 1024);
    // (== bytes_for(f.S))
    return f;
}

// Backward workspace: header (error word, ticket) | tile counters of the
// fused schedule | one wave of bf16 dZ [chunk, Vp].
struct BwdLayout {
    int64_t Vp;
    int Vt, Mt_max;
    size_t off_cnt, cnt_bytes, off_dz;
};

BwdLayout bwd_layout(int64_t M, int64_t V) {
    BwdLayout L{};
    L.Vp = cdiv(V, BN) * BN;
    L.Vt = static_cast<int>(L.Vp / BN);
    L.Mt_max = static_cast<int>(std::max<int64_t>(1, cdiv(M, PM)));
    L.off_cnt = kHeaderBytes;
    L.cnt_bytes = align_up((2 * static_cast<size_t>(L.Mt_max) + 2 * static_cast<size_t>(L.Vt)) * 4, 1024);
    L.off_dz = L.off_cnt + L.cnt_bytes;
    return L;
}

size_t backward_bytes(int64_t M, int64_t V, int64_t chunk_rows) {
    const BwdLayout L = bwd_layout(M, V);
    const int64_t mr = std::max<int64_t>(BM, cdiv(M, BM) * BM);
    int64_t c = chunk_rows > 0 ? chunk_rows : kDefaultChunkRows;
    c = std::max<int64_t>(BM, cdiv(c, BM) * BM);
    c = std::min(c, mr);
    return L.off_dz + static_cast<size_t>(c) * L.Vp * 2;
}

// The wave size and schedule a backward call runs with.  Split waves are any
// multiple of 128 rows; fused waves are all rows (one wave) or a multiple of
// 256 rows, so no 256-row pair tile straddles two waves.
struct BwdChoice {
    flp_bwd_schedule schedule;
    int64_t chunk;   // rows of a row wave (all rows, rounded up to 128, for FLP_BWD_VSPLIT)
    int64_t waves;   // row waves, or vocabulary chunks for FLP_BWD_VSPLIT
    int64_t vc;      // padded vocabulary columns per chunk (all of them unless FLP_BWD_VSPLIT)
    size_t off_scr;  // FLP_BWD_VSPLIT: fp32 dX scratch [M, H] (0: none)
    size_t off_dz;   // the bf16 dZ buffer [chunk rows, vc]
};

flp_status choose_backward(int64_t M, int64_t H, int64_t V, size_t workspace_bytes, flp_bwd_schedule want,
                           BwdChoice* out) {
    if (want != FLP_BWD_AUTO && want != FLP_BWD_SPLIT && want != FLP_BWD_FUSED && want != FLP_BWD_VSPLIT)
        return fail(FLP_ERR_INVALID_ARG,
                    "schedule must be FLP_BWD_AUTO, FLP_BWD_SPLIT, FLP_BWD_FUSED or FLP_BWD_VSPLIT");
    const BwdLayout L = bwd_layout(M, V);
    if (workspace_bytes < L.off_dz) return fail(FLP_ERR_WORKSPACE, "backward workspace too small");
    const int64_t mr = std::max<int64_t>(BM, cdiv(M, BM) * BM);
    // the vocabulary-split plan: all rows in one wave, the vocabulary in
    // chunks of vc columns; dX accumulates over the chunks in an fp32 scratch
    const size_t scr = align_up(static_cast<size_t>(std::max<int64_t>(M, 1)) * H * 4, 1024);
    const size_t vs_off_dz = L.off_dz + scr;
    const int64_t vs_vc =
        workspace_bytes < vs_off_dz
            ? 0
            : std::min<int64_t>(L.Vp, static_cast<int64_t>((workspace_bytes - vs_off_dz) /
                                                             (static_cast<size_t>(mr) * 2)) / BN * BN);
    auto take_vsplit = [&]() {
        out->schedule = FLP_BWD_VSPLIT;
        out->chunk = mr;
        out->waves = M > 0 ? cdiv(L.Vp, vs_vc) : 0;
        out->vc = vs_vc;
        out->off_scr = L.off_dz;
        out->off_dz = vs_off_dz;
        return FLP_OK;
    };
    if (want == FLP_BWD_VSPLIT) {
        if (workspace_bytes < vs_off_dz)
            return fail(FLP_ERR_WORKSPACE, "backward workspace has no room for the fp32 dX scratch");
        if (vs_vc < BN)
            return fail(FLP_ERR_WORKSPACE, "backward workspace holds fewer than 256 vocabulary columns of dZ");
        return take_vsplit();
    }
    const int64_t fit = static_cast<int64_t>((workspace_bytes - L.off_dz) / (static_cast<size_t>(L.Vp) * 2));
    const int64_t split_chunk = std::min(mr, fit / BM * BM);
    // Short row waves make every dW tile short (K = wave rows) and re-add dW
    // once per wave; below 2048-row waves the vocabulary-split plan measured
    // faster on GB300 (+10 % at 1024-row waves, +50 % at 512), above it the
    // split schedule (its dX tiles run the whole vocabulary as K).
    const bool short_waves = fit / BM * BM < std::min<int64_t>(mr, 2048);
    if (want == FLP_BWD_AUTO && short_waves && vs_vc >= BN) return take_vsplit();
    if (split_chunk < BM) return fail(FLP_ERR_WORKSPACE, "backward workspace holds fewer than 128 rows of dZ");
    const int64_t fused_chunk = fit >= mr ? mr : fit / PM * PM;
    const int64_t fused_waves = fused_chunk > 0 ? cdiv(std::max<int64_t>(M, 1), fused_chunk) : 0;
    // the fused counters' cumulative targets must fit 32 bits
    const bool fused_ok = fused_chunk >= PM || fused_chunk == mr;
    const bool fused_fits = fused_ok && static_cast<double>(L.Vt) * fused_waves * 2.0 < 4.0e9;
    // On GB300 the split schedule measured faster at every shape tried: the
    // chip runs at its power cap, and a launch that mixes dZ tiles (exp-heavy
    // epilogue) with dX / dW tiles runs at a lower clock for the same cycles
    // per tile, which costs more than the launch boundaries it removes.
    const flp_bwd_schedule use = want == FLP_BWD_AUTO ? FLP_BWD_SPLIT : want;
    if (use == FLP_BWD_FUSED && !fused_fits)
        return fail(FLP_ERR_UNSUPPORTED,
                    "the fused backward needs a workspace that holds all rows of dZ or at least 256 rows");
    out->schedule = use;
    out->chunk = use == FLP_BWD_FUSED ? fused_chunk : split_chunk;
    out->waves = M > 0 ? cdiv(M, out->chunk) : 0;
    out->vc = L.Vp;
    out->off_scr = 0;
    out->off_dz = L.off_dz;
    return FLP_OK;
}

bool smem_attrs_done(DevInfo* d) { return d->attrs_set; }

template <bool kEnt>
cudaError_t set_fwd_smem_attr() {
    return cudaFuncSetAttribute(flp_fwd_kernel<kEnt>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SMEM_ALLOC);
}

flp_status ensure_attrs(DevInfo* d) {
    if (smem_attrs_done(d)) return FLP_OK;
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = set_fwd_smem_attr<true>();
    if (e == cudaSuccess) e = set_fwd_smem_attr<false>();
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(flp_dz_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(flp_bwd_kernel<kHasDx | kHasDw>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_ALLOC);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(flp_bwd_kernel<kHasDz | kHasDx | kHasDw>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    // How many clusters of two fit at once (SMs that a cluster cannot pair up
    // stay idle); the persistent grids never exceed it.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(d->sm_count));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, flp_fwd_kernel<true>, &cfg);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
    if (clusters < 1) return fail(FLP_ERR_UNSUPPORTED, "no CTA pair fits on the device");
    std::lock_guard<std::mutex> lk(g_mu);
    d->pairs = std::min(clusters, std::max(1, d->sm_count / 2));
    d->attrs_set = true;
    return FLP_OK;
}

flp_status check_device(DevInfo** d) {
    flp_status st = device_info(d, nullptr);
    if (st != FLP_OK) return st;
    if ((*d)->major != 10 || (*d)->minor != 3)
        return fail(FLP_ERR_UNSUPPORTED, "kernels are built for sm_103a (GB300) only");
    return ensure_attrs(*d);
}

// A device pointer must live on the device the call launches on (the one
// current on the calling thread); host or managed-elsewhere memory is refused.
flp_status check_on_current_device(const void* p, const char* what) {
    if (!p) return FLP_OK;
    int dev = 0;
    FLP_CUDA(cudaGetDevice(&dev));
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) {
        char buf[160];
        snprintf(buf, sizeof buf, "%s is not device memory", what);
        return fail(FLP_ERR_INVALID_ARG, buf);
    }
    if (a.type == cudaMemoryTypeDevice && a.device != dev) {
        char buf[160];
        snprintf(buf, sizeof buf, "%s lives on device %d but the current device is %d", what, a.device, dev);
        return fail(FLP_ERR_INVALID_ARG, buf);
    }
    return FLP_OK;
}

// Launches `kernel` on `grid` CTAs grouped in clusters of two (the CTA pairs
// that share each tcgen05.mma.cta_group::2 tile).  With `after_kernel` the
// launch follows another of this library's kernels on the stream and uses
// programmatic dependent launch: its CTAs may be scheduled on the SMs the
// previous grid frees while that grid's last tiles finish, run their set-up,
// and wait in griddepcontrol.wait for its results.
template <typename... KArgs, typename... Args>
flp_status launch_pairs_n(void (*kernel)(KArgs...), int grid, int threads, cudaStream_t s, const char* what,
                          bool after_kernel, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_kernel ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, what);
    return FLP_OK;
}

template <typename... KArgs, typename... Args>
flp_status launch_pairs(void (*kernel)(KArgs...), int grid, cudaStream_t s, const char* what, bool after_kernel,
                        Args&&... args) {
    return launch_pairs_n(kernel, grid, NUM_THREADS, s, what, after_kernel, std::forward<Args>(args)...);
}

template <bool kEnt>
flp_status launch_fwd(int grid, const CUtensorMap& a, const CUtensorMap& b, const FwdParams& p,
                      cudaStream_t s) {
    return launch_pairs_n(flp_fwd_kernel<kEnt>, grid, WIDE_THREADS, s, "flp_fwd_kernel launch", false, a, b, p);
}

flp_status common_checks(const void* X, const void* W, const int64_t* targets, int64_t M,
                         int64_t H, int64_t V) {
    if (M < 0 || H < 1 || V < 1) return fail(FLP_ERR_INVALID_ARG, "M >= 0, H >= 1 and V >= 1 required");
    if (H % 8 != 0) return fail(FLP_ERR_UNSUPPORTED, "H must be a multiple of 8 (TMA row pitch)");
    if (M > (int64_t)INT_MAX - BM || V > (int64_t)INT_MAX - BN || H > (int64_t)INT_MAX - BN)
        return fail(FLP_ERR_UNSUPPORTED, "dimension too large for int32 tile coordinates");
    if (M == 0) return FLP_OK;  // nothing is read: empty inputs may be null
    if (!X || !W || !targets) return fail(FLP_ERR_INVALID_ARG, "X, W and targets must be non-null");
    if (!aligned16(X) || !aligned16(W) || !aligned16(targets))
        return fail(FLP_ERR_INVALID_ARG, "X, W and targets must be 16-byte aligned");
    return FLP_OK;
}

// The forward's two launches for plan f, its scratch (header with the error
// word, per-split partials, target logits) at ws: the header is cleared, the
// tile kernel writes the raw partials, the merge the outputs.  Shared by the
// workspace forward, the allocation-free forward and the wait self-test, so
// that their results come from the same code.
flp_status launch_forward(const void* X, const void* W, const int64_t* targets, int64_t M, int64_t H,
                          int64_t V, int64_t ignore_index, float scale, int ent, float* logprob,
                          float* lse, float* entropy, const FwdPlan& f, uint8_t* ws,
                          unsigned long long wait_limit_ns, int debug_stall_after, cudaStream_t s) {
    int* err = reinterpret_cast<int*>(ws);
    FLP_CUDA(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
    if (M == 0) return FLP_OK;

    CUtensorMap tmX, tmW;
    flp_status st = tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, H, M, H * 2, BK, BM);
    if (st != FLP_OK) return st;
    st = tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, BK, BNH);
    if (st != FLP_OK) return st;

    FwdParams p{};
    p.units = f.units;
    p.Mt = f.Mt;
    p.Nt = f.Vt;
    p.S = f.S;
    p.tps = f.tps;
    p.GM = f.GM;
    p.KB = static_cast<int>(cdiv(H, BK));
    p.M = static_cast<int>(M);
    p.V = static_cast<int>(V);
    p.ignore_index = ignore_index;
    p.scale = scale;
    p.scale2 = scale * LOG2E;
    p.y = reinterpret_cast<const long long*>(targets);
    p.part_m = reinterpret_cast<float*>(ws + f.off_m);
    p.part_s = reinterpret_cast<float*>(ws + f.off_s);
    p.part_t = ent ? reinterpret_cast<float*>(ws + f.off_t) : nullptr;
    p.zy = reinterpret_cast<float*>(ws + f.off_zy);
    p.err = err;
    p.wait_limit_ns = wait_limit_ns;
    p.debug_stall_after = debug_stall_after;
    mark(0, s);
    st = ent ? launch_fwd<true>(f.grid, tmX, tmW, p, s) : launch_fwd<false>(f.grid, tmX, tmW, p, s);
    if (st != FLP_OK) return st;
    mark(1, s);

    MergeParams mp{};
    mp.M = static_cast<int>(M);
    mp.S = 2 * f.S;  // two 256-column halves per split
    mp.V = static_cast<int>(V);
    mp.ignore_index = ignore_index;
    mp.compute_entropy = ent;
    mp.y = p.y;
    mp.part_m = p.part_m;
    mp.part_s = p.part_s;
    mp.part_t = p.part_t;
    mp.zy = p.zy;
    mp.logprob = logprob;
    mp.lse = lse;
    mp.entropy = entropy;
    mp.err = err;
    mark(2, s);
    {
        // programmatic dependent launch on the tile kernel (unless an event
        // recorded in between separates them)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(cdiv(M, MERGE_ROWS)));
        cfg.blockDim = dim3(MERGE_ROWS * MERGE_WAYS);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, flp_merge_kernel, mp);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "flp_merge_kernel launch");
    }
    mark(3, s);
    return FLP_OK;
}

// Argument checks shared by both forward entry points.
flp_status forward_checks(const void* X, const void* W, const int64_t* targets, int64_t M, int64_t H,
                          int64_t V, float scale, int ent, const float* logprob, const float* lse,
                          const float* entropy) {
    flp_status st = common_checks(X, W, targets, M, H, V);
    if (st != FLP_OK) return st;
    if (M > 0 && (!logprob || !lse || (ent && !entropy) || (!ent && entropy)))
        return fail(FLP_ERR_INVALID_ARG, "logprob and lse required; entropy iff compute_entropy");
    if (!aligned16(logprob) || !aligned16(lse) || (entropy && !aligned16(entropy)))
        return fail(FLP_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(FLP_ERR_INVALID_ARG, "scale must be finite");
    return FLP_OK;
}

}  // namespace

// =================================================================== C ABI

extern "C" {

const char* flp_status_string(flp_status s) {
    switch (s) {
        case FLP_OK: return "ok";
        case FLP_ERR_INVALID_ARG: return "invalid argument";
        case FLP_ERR_UNSUPPORTED: return "unsupported shape or device";
        case FLP_ERR_WORKSPACE: return "workspace missing or too small";
        case FLP_ERR_CUDA: return "CUDA error";
        case FLP_ERR_BAD_TARGET: return "target outside [0, V) that is not ignore_index";
        case FLP_ERR_TIMEOUT: return "a kernel wait timed out";
    }
    return "unknown status";
}

const char* flp_last_error_message(void) { return g_msg.c_str(); }

flp_status flp_set_phase_events(void* const* events, int count) {
    if (count < 0 || count > kMaxPhaseEvents)
        return fail(FLP_ERR_INVALID_ARG, "count must be in [0, 10]");
    g_num_events = events ? count : 0;
    for (int i = 0; i < kMaxPhaseEvents; ++i) g_events[i] = (events && i < count) ? events[i] : nullptr;
    return FLP_OK;
}

flp_status flp_workspace_query(int64_t M, int64_t H, int64_t V, int compute_entropy,
                               size_t* fwd_bytes, size_t* bwd_bytes) {
    return flp_workspace_query_ex(M, H, V, compute_entropy, 0, fwd_bytes, bwd_bytes);
}

flp_status flp_workspace_query_ex(int64_t M, int64_t H, int64_t V, int compute_entropy,
                                  int64_t chunk_rows, size_t* fwd_bytes, size_t* bwd_bytes) {
    if (M < 0 || H < 1 || V < 1) return fail(FLP_ERR_INVALID_ARG, "M >= 0, H >= 1 and V >= 1 required");
    DevInfo* d;
    flp_status st = check_device(&d);
    if (st != FLP_OK) return st;
    if (fwd_bytes) *fwd_bytes = plan_forward(M, H, V, compute_entropy ? 1 : 0, d->pairs).bytes;
    if (bwd_bytes) *bwd_bytes = backward_bytes(M, V, chunk_rows);
    return FLP_OK;
}

flp_status flp_forward(const void* X, const void* W, const int64_t* targets, int64_t M,
                       int64_t H, int64_t V, int64_t ignore_index, float scale,
                       int compute_entropy, float* logprob, float* lse, float* entropy,
                       void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange range("flp_forward");
    const int ent = compute_entropy ? 1 : 0;
    flp_status st = forward_checks(X, W, targets, M, H, V, scale, ent, logprob, lse, entropy);
    if (st != FLP_OK) return st;
    DevInfo* d;
    st = check_device(&d);
    if (st != FLP_OK) return st;
    if (M > 0 && (st = check_on_current_device(X, "X")) != FLP_OK) return st;
    const FwdPlan f = plan_forward(M, H, V, ent, d->pairs);
    if (!workspace || workspace_bytes < f.bytes || !aligned16(workspace))
        return fail(FLP_ERR_WORKSPACE, "forward workspace null, misaligned or too small");
    return launch_forward(X, W, targets, M, H, V, ignore_index, scale, ent, logprob, lse, entropy, f,
                          static_cast<uint8_t*>(workspace), kWaitLimitNs, -1,
                          static_cast<cudaStream_t>(stream));
}

flp_status flp_backward_plan(int64_t M, int64_t H, int64_t V, size_t workspace_bytes,
                             flp_bwd_schedule schedule, int64_t* wave_rows, int64_t* waves,
                             flp_bwd_schedule* schedule_used) {
    if (M < 0 || H < 1 || V < 1) return fail(FLP_ERR_INVALID_ARG, "M >= 0, H >= 1 and V >= 1 required");
    BwdChoice c{};
    flp_status st = choose_backward(M, H, V, workspace_bytes, schedule, &c);
    if (st != FLP_OK) return st;
    if (wave_rows) *wave_rows = c.chunk;
    if (waves) *waves = c.waves;
    if (schedule_used) *schedule_used = c.schedule;
    return FLP_OK;
}

flp_status flp_backward(const void* X, const void* W, const int64_t* targets, int64_t M,
                        int64_t H, int64_t V, int64_t ignore_index, float scale,
                        int compute_entropy, const float* lse, const float* entropy,
                        const float* grad_logprob, const float* grad_entropy, void* dX,
                        flp_dtype dX_dtype, void* dW, flp_dtype dW_dtype, int accumulate_dW,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return flp_backward_ex(X, W, targets, M, H, V, ignore_index, scale, compute_entropy, lse, entropy,
                           grad_logprob, grad_entropy, dX, dX_dtype, dW, dW_dtype, accumulate_dW,
                           workspace, workspace_bytes, FLP_BWD_AUTO, stream);
}

}  // extern "C"

namespace {

// Appends segments to a launch's schedule (BwdParams::seg).
struct SegList {
    BwdParams* p;
    bool overflow = false;
    void add(int kind, int wave, int a0, int an, int b0, int lag, int64_t count) {
        if (count <= 0) return;
        if (p->nseg >= MAX_SEGS || static_cast<int64_t>(p->total) + count > INT_MAX / 2) {
            overflow = true;
            return;
        }
        BwdSeg& g = p->seg[p->nseg++];
        g.start = p->total;
        g.kind = kind;
        g.wave = wave;
        g.a0 = a0;
        g.an = an;
        g.b0 = b0;
        g.lag = lag;
        p->total += static_cast<int>(count);
    }
    // dX tiles of row tiles [m0, m0 + gm) in groups of 8 rows (hidden tiles
    // outer inside a group): the pairs running together share dZ rows and W
    // columns in L2.  Wide (256 x 512) when H spans an even number of
    // 256-column tiles (see dx_wide).
    void dx_rows(int wave, int m0, int gm, int Nh, int KB) {
        const bool wide = dx_wide(Nh, KB);
        for (int s = m0; s < m0 + gm; s += 8) {
            const int n = std::min(8, m0 + gm - s);
            add(wide ? kSegDx2 : kSegDx, wave, s, n, 0, 0, static_cast<int64_t>(n) * dx_per_row(Nh, KB));
        }
    }
    // A wide tile's epilogue cannot overlap the next tile's MMAs (it holds
    // both accumulators), yet even on a 64-block K loop (4096-column chunks
    // of the vocabulary split) wide tiles measured 13 % more work per clock
    // than pairs of 256-column tiles, so the K length does not enter.
    static bool dx_wide(int Nh, int /*KB*/) { return Nh % 2 == 0; }
    static int dx_per_row(int Nh, int KB) { return dx_wide(Nh, KB) ? Nh / 2 : Nh; }
};

constexpr int kDwLag = 8;  // vocabulary tiles between a dZ column and the dW column paired with it

// The fused schedule of one wave (see bwd.cuh).  Row tiles are swept in
// groups of GM (vocabulary outer, so each W tile is shared by the group);
// the dX tiles of a group follow once a few columns of the next group have
// been handed out; during the last group's sweep, each dZ column is followed
// by the dW tiles of the column kDwLag tiles earlier; then come a buffer of
// dW tiles (time for the sweep's last stores), the last group's dX tiles
// (long: K = padded vocabulary) and the remaining dW tiles (short), enough of
// them to even out the end of the dX tiles.
void fused_wave_schedule(SegList& sl, int w, int Mt, int GM, int Vt, int Nh, int pairs, int KB_v,
                         int KB_dw, bool more_waves) {
    const int G = static_cast<int>(cdiv(Mt, GM));
    const int lead = 3 * pairs;  // tickets handed out before a dependent unit
    for (int g = 0; g < G; ++g) {
        const int m0 = g * GM, gm = std::min(GM, Mt - m0);
        int c = 0;
        if (g > 0) {
            const int Lc = static_cast<int>(std::min<int64_t>(Vt, cdiv(lead, gm)));
            sl.add(kSegDz, w, m0, gm, 0, 0, static_cast<int64_t>(gm) * Lc);
            sl.dx_rows(w, (g - 1) * GM, GM, Nh, KB_v);
            c = Lc;
        }
        if (g < G - 1) {
            sl.add(kSegDz, w, m0, gm, c, 0, static_cast<int64_t>(gm) * (Vt - c));
            continue;
        }
        const int dx_len = KB_v * (SegList::dx_wide(Nh, KB_v) ? 2 : 1);  // K blocks x sub-tiles of a dX tile
        const double tail_units =
            static_cast<double>(pairs) * dx_len / std::max(1, KB_dw) * (more_waves ? 1.25 : 1.0);
        const int Ct = static_cast<int>(std::min<double>(Vt, std::ceil(tail_units / Nh)));
        const int Cb = static_cast<int>(std::min<int64_t>(Vt - Ct, cdiv(lead, Nh)));
        const int z0 = std::max(c, Ct + Cb + kDwLag);  // first dZ column paired with a dW column
        if (z0 < Vt) {
            sl.add(kSegDz, w, m0, gm, c, 0, static_cast<int64_t>(gm) * (z0 - c));
            sl.add(kSegDzDw, w, m0, gm, z0, kDwLag, static_cast<int64_t>(gm + Nh) * (Vt - z0));
            sl.add(kSegDw, w, 0, 0, Ct, 0, static_cast<int64_t>(Cb) * Nh);
            sl.dx_rows(w, m0, gm, Nh, KB_v);
            sl.add(kSegDw, w, 0, 0, 0, 0, static_cast<int64_t>(Ct) * Nh);
            sl.add(kSegDw, w, 0, 0, Ct + Cb, 0, static_cast<int64_t>(z0 - kDwLag - Ct - Cb) * Nh);
            sl.add(kSegDw, w, 0, 0, Vt - kDwLag, 0, static_cast<int64_t>(kDwLag) * Nh);
        } else {
            sl.add(kSegDz, w, m0, gm, c, 0, static_cast<int64_t>(gm) * (Vt - c));
            sl.add(kSegDw, w, 0, 0, Ct, 0, static_cast<int64_t>(Cb) * Nh);
            sl.dx_rows(w, m0, gm, Nh, KB_v);
            sl.add(kSegDw, w, 0, 0, 0, 0, static_cast<int64_t>(Ct) * Nh);
            sl.add(kSegDw, w, 0, 0, Ct + Cb, 0, static_cast<int64_t>(Vt - Ct - Cb) * Nh);
        }
    }
}

// One launch of flp_bwd_kernel: the rows its row tensor maps cover and its
// schedule (the segment fields of BwdParams; the rest is filled per call).
struct LaunchSpec {
    int64_t r0, rows, dz_rows;  // X / dX maps over rows [r0, r0 + rows); dZ buffer rows
    int64_t dz_cols;            // dZ buffer columns (the padded vocabulary, or one chunk of it)
    int mark_begin, mark_end;   // phase events recorded around the launch (-1: none)
    BwdParams p;
};

// Every launch of a backward call, in stream order.
flp_status plan_backward_launches(int64_t M, int64_t H, int64_t V, const BwdChoice& ch, int pairs,
                                  int accumulate_dW, std::vector<LaunchSpec>& out) {
    out.clear();
    const int Vt = static_cast<int>(cdiv(V, BN));
    const int Nh = static_cast<int>(cdiv(H, BN));
    const int KB_v = Vt * (BN / BK);
    const int gm_rows = static_cast<int>(std::max<int64_t>(4, 40ll * 1000 * 1000 / (PM * 2 * H)));
    const int64_t chunk = ch.chunk;
    // One wave's two launches over vocabulary tiles [vt0, vt1): its dZ tiles
    // (static order), then its dX and dW tiles.
    auto add_pair = [&](int64_t r0, int64_t rows, int64_t dz_rows, int vt0, int vt1, bool first,
                        bool dx_add, bool dw_add) -> flp_status {
        LaunchSpec a{};
        a.r0 = r0;
        a.rows = rows;
        a.dz_rows = dz_rows;
        a.dz_cols = ch.vc;
        a.p.Vt = Vt;
        a.p.Nh = Nh;
        a.p.KB_v = (vt1 - vt0) * (BN / BK);
        a.p.Ndx = SegList::dx_per_row(Nh, a.p.KB_v);
        a.p.vt0 = vt0;
        a.p.vt_end = vt1;
        a.p.M = static_cast<int>(rows);
        a.p.chunk = static_cast<int>(rows);
        a.p.nwaves = 1;
        a.p.Mt_full = static_cast<int>(cdiv(rows, PM));
        a.p.deps = 0;
        a.p.dw_add0 = dw_add ? 1 : 0;
        const int Mt = a.p.Mt_full;
        const int GM = std::min(Mt, gm_rows);
        LaunchSpec b = a;
        b.p.dx_add = dx_add ? 1 : 0;
        a.p.static_order = 1;  // equal-length wide dZ tiles: static round-robin (flp_dz_kernel)
        a.mark_begin = first ? 4 : -1;
        a.mark_end = first ? 5 : -1;
        b.mark_begin = first ? 6 : -1;
        b.mark_end = first ? 7 : -1;
        SegList dzs{&a.p};
        const int nw = (vt1 - vt0 + 1) / 2;  // 512-column dZ tiles per row tile
        for (int m0 = 0; m0 < Mt; m0 += GM) {
            const int gm = std::min(GM, Mt - m0);
            dzs.add(kSegDz2, 0, m0, gm, vt0, 0, static_cast<int64_t>(gm) * nw);
        }
        SegList gl{&b.p};
        gl.dx_rows(0, 0, Mt, Nh, a.p.KB_v);
        // dW tiles wide (256 x 512) when H spans an even number of 256-column tiles
        if (Nh % 2 == 0)
            gl.add(kSegDw2, 0, 0, 0, vt0, 0, static_cast<int64_t>(vt1 - vt0) * (Nh / 2));
        else
            gl.add(kSegDw, 0, 0, 0, vt0, 0, static_cast<int64_t>(vt1 - vt0) * Nh);
        if (dzs.overflow || gl.overflow) return fail(FLP_ERR_UNSUPPORTED, "backward schedule too large");
        out.push_back(a);
        out.push_back(b);
        return FLP_OK;
    };
    if (ch.schedule == FLP_BWD_SPLIT) {
        for (int64_t r0 = 0; r0 < M; r0 += chunk) {
            const int64_t rows = std::min(chunk, M - r0);
            flp_status st = add_pair(r0, rows, rows, 0, Vt, r0 == 0, false, accumulate_dW || r0 > 0);
            if (st != FLP_OK) return st;
        }
        return FLP_OK;
    }
    if (ch.schedule == FLP_BWD_VSPLIT) {
        // one wave of all rows; each dW tile is written once (its chunk holds all its K)
        const int tpc = static_cast<int>(ch.vc / BN);  // vocabulary tiles per chunk
        for (int vt0 = 0; vt0 < Vt; vt0 += tpc) {
            flp_status st = add_pair(0, M, chunk, vt0, std::min(Vt, vt0 + tpc), vt0 == 0, vt0 > 0,
                                     accumulate_dW != 0);
            if (st != FLP_OK) return st;
        }
        return FLP_OK;
    }
    // fused: every wave in as few launches as the segment table allows (normally one)
    const int nwaves = static_cast<int>(ch.waves);
    const int Mt_full = static_cast<int>(cdiv(chunk, PM));
    const int GM = std::min(Mt_full, gm_rows);
    int w = 0;
    while (w < nwaves) {
        LaunchSpec L{};
        L.r0 = 0;
        L.rows = M;
        L.dz_rows = chunk;
        L.dz_cols = ch.vc;
        L.mark_begin = (w == 0) ? 4 : -1;
        L.mark_end = -1;
        L.p.Vt = Vt;
        L.p.Nh = Nh;
        L.p.Ndx = SegList::dx_per_row(Nh, KB_v);
        L.p.KB_v = KB_v;
        L.p.M = static_cast<int>(M);
        L.p.chunk = static_cast<int>(chunk);
        L.p.nwaves = nwaves;
        L.p.Mt_full = Mt_full;
        L.p.deps = 1;
        L.p.dw_add0 = accumulate_dW ? 1 : 0;
        int w_end = w;
        while (w_end < nwaves) {
            const int nseg0 = L.p.nseg, total0 = L.p.total;
            SegList sl{&L.p};
            const int64_t rows = std::min(chunk, M - static_cast<int64_t>(w_end) * chunk);
            fused_wave_schedule(sl, w_end, static_cast<int>(cdiv(rows, PM)), GM, Vt, Nh, pairs, KB_v,
                                static_cast<int>(cdiv(rows, BK)), w_end + 1 < nwaves);
            if (sl.overflow) {
                if (w_end == w) return fail(FLP_ERR_UNSUPPORTED, "backward schedule too large");
                L.p.nseg = nseg0;  // this wave starts the next launch
                L.p.total = total0;
                break;
            }
            ++w_end;
        }
        if (w_end == nwaves) L.mark_end = 5;
        out.push_back(L);
        w = w_end;
    }
    return FLP_OK;
}

struct BwdMaps {
    CUtensorMap Xk, Wk, Dz, Wmn, DzMn, Xmn, Dx, Dw;
    CUtensorMap DzSt;  // dZ buffer: the wide dZ tiles' 32-column store boxes (64-byte swizzle)
};

// The tile kinds (kHasDz | kHasDx | kHasDw) a launch's segments hold.
int launch_kinds(const BwdParams& p) {
    int k = 0;
    for (int i = 0; i < p.nseg; ++i) {
        switch (p.seg[i].kind) {
            case kSegDz: k |= kHasDz; break;
            case kSegDz2: k |= kHasDzWide; break;
            case kSegDx:
            case kSegDx2: k |= kHasDx; break;
            case kSegDw:
            case kSegDw2: k |= kHasDw; break;
            default: k |= kHasDz | kHasDw; break;
        }
    }
    return k;
}

// after_kernel: the launch directly follows another of this library's kernels
// on the stream (programmatic dependent launch, see launch_pairs_n).
// narrow: the dX / dW store maps have narrow (64-byte) boxes, which only the
// two-group dX + dW instantiation writes.
flp_status launch_bwd(int pairs, const BwdMaps& m, const BwdParams& p, unsigned long long* ticket_base,
                      cudaStream_t s, bool after_kernel = false, bool narrow = false) {
    const int np = std::min(p.total, pairs);
    // a ticketed launch draws every unit plus one past the end per CTA pair;
    // a static round-robin draws none
    if (!p.static_order) *ticket_base += static_cast<unsigned long long>(p.total) + np;
    const char* what = "flp_bwd_kernel launch";
    switch (launch_kinds(p)) {
        case kHasDzWide:
            return launch_pairs_n(flp_dz_kernel, 2 * np, WIDE_THREADS, s, "flp_dz_kernel launch", after_kernel,
                                  m.Xk, m.Wk, m.DzSt, p);
        case kHasDx | kHasDw:
            if (!narrow) return fail(FLP_ERR_UNSUPPORTED, "dX + dW launch without narrow store maps");
            return launch_pairs_n(flp_bwd_kernel<kHasDx | kHasDw>, 2 * np, WIDE_THREADS, s, what, after_kernel,
                                  m.Xk, m.Wk, m.Dz, m.Wmn, m.DzMn, m.Xmn, m.Dx, m.Dw, p);
        default:
            if (narrow) return fail(FLP_ERR_UNSUPPORTED, "backward launch of this kind with narrow store maps");
            return launch_pairs(flp_bwd_kernel<kHasDz | kHasDx | kHasDw>, 2 * np, s, what, after_kernel, m.Xk,
                                m.Wk, m.Dz, m.Wmn, m.DzMn, m.Xmn, m.Dx, m.Dw, p);
    }
}

}  // namespace

extern "C" {

flp_status flp_backward_ex(const void* X, const void* W, const int64_t* targets, int64_t M,
                           int64_t H, int64_t V, int64_t ignore_index, float scale,
                           int compute_entropy, const float* lse, const float* entropy,
                           const float* grad_logprob, const float* grad_entropy, void* dX,
                           flp_dtype dX_dtype, void* dW, flp_dtype dW_dtype, int accumulate_dW,
                           void* workspace, size_t workspace_bytes, flp_bwd_schedule schedule,
                           void* stream) {
    NvtxRange range("flp_backward");
    flp_status st = common_checks(X, W, targets, M, H, V);
    if (st != FLP_OK) return st;
    const int ent = compute_entropy ? 1 : 0;
    if ((M > 0 && !dX) || !dW) return fail(FLP_ERR_INVALID_ARG, "dX and dW must be non-null");
    if (dX_dtype != FLP_BF16 && dX_dtype != FLP_F32)
        return fail(FLP_ERR_INVALID_ARG, "dX_dtype must be FLP_BF16 or FLP_F32");
    if (dW_dtype != FLP_F32 && dW_dtype != FLP_BF16)
        return fail(FLP_ERR_INVALID_ARG, "dW_dtype must be FLP_F32 or FLP_BF16");
    if (dW_dtype == FLP_BF16 && accumulate_dW)
        return fail(FLP_ERR_UNSUPPORTED, "a bf16 dW cannot be accumulated into (fp32 accumulation); use an fp32 dW");
    if (M > 0 && (!lse || (ent && !entropy)))
        return fail(FLP_ERR_INVALID_ARG, "lse (and entropy when compute_entropy) required");
    if (!aligned16(dX) || !aligned16(dW) || (lse && !aligned16(lse)) ||
        (entropy && !aligned16(entropy)) || (grad_logprob && !aligned16(grad_logprob)) ||
        (grad_entropy && !aligned16(grad_entropy)))
        return fail(FLP_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(FLP_ERR_INVALID_ARG, "scale must be finite");
    DevInfo* d;
    st = check_device(&d);
    if (st != FLP_OK) return st;
    if (M > 0 && (st = check_on_current_device(X, "X")) != FLP_OK) return st;
    if (!workspace || !aligned16(workspace))
        return fail(FLP_ERR_WORKSPACE, "backward workspace null or misaligned");
    BwdChoice ch{};
    if ((st = choose_backward(M, H, V, workspace_bytes, schedule, &ch)) != FLP_OK) return st;
    const int64_t chunk = ch.chunk;
    if (dW_dtype == FLP_BF16 && chunk < M)
        return fail(FLP_ERR_UNSUPPORTED,
                    "a bf16 dW needs the backward in one wave (waves accumulate dW in fp32): pass a "
                    "workspace that holds all M rows of dZ, or an fp32 dW");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* err = reinterpret_cast<int*>(ws);
    FLP_CUDA(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
    const size_t dx_es = dX_dtype == FLP_F32 ? 4 : 2;
    const size_t dw_es = dW_dtype == FLP_F32 ? 4 : 2;
    const bool no_grad = (grad_logprob == nullptr) && (!ent || grad_entropy == nullptr);
    if (M == 0 || no_grad) {
        if (M > 0) FLP_CUDA(cudaMemsetAsync(dX, 0, static_cast<size_t>(M) * H * dx_es, s));
        if (!accumulate_dW) FLP_CUDA(cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * H * dw_es, s));
        return FLP_OK;
    }
    const BwdLayout L = bwd_layout(M, V);
    uint8_t* dz = ws + ch.off_dz;
    const int pairs = d->pairs;
    unsigned long long ticket_base = 0;
    // The vocabulary-split schedule accumulates a bf16 dX over its chunks in
    // the fp32 scratch, then rounds it once.
    const bool dx_scratch = ch.schedule == FLP_BWD_VSPLIT && ch.waves > 1 && dX_dtype == FLP_BF16;
    float* scr = dx_scratch ? reinterpret_cast<float*>(ws + ch.off_scr) : nullptr;

    BwdMaps m{};
    // the split and vocabulary-split schedules' dX + dW launches store through
    // narrow boxes (two epilogue groups); the fused launch through 128-byte ones
    const bool narrow = ch.schedule != FLP_BWD_FUSED;
    const CUtensorMapSwizzle out_swz = narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const uint32_t box_bf16 = narrow ? 32 : 64, box_f32 = narrow ? 16 : 32;  // columns per store box
    if ((st = tmap_2d(&m.Wk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, BK, BNH)) != FLP_OK) return st;
    if ((st = tmap_2d(&m.Wmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, 64, 64)) != FLP_OK) return st;
    if (dW_dtype == FLP_BF16)
        st = tmap_2d(&m.Dw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dW, H, V, H * 2, box_bf16, BM, out_swz);
    else
        st = tmap_2d(&m.Dw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dW, H, V, H * 4, box_f32, BM, out_swz);
    if (st != FLP_OK) return st;

    // Row tensor maps (X, dX, dZ buffer) over `rows` rows starting at global
    // row r0; the dZ buffer is dz_rows x dz_cols.
    auto row_maps = [&](int64_t r0, int64_t rows, int64_t dz_rows, int64_t dz_cols) -> flp_status {
        const uint8_t* Xc = static_cast<const uint8_t*>(X) + r0 * H * 2;
        flp_status e;
        if ((e = tmap_2d(&m.Xk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xc, H, rows, H * 2, BK, BM)) != FLP_OK) return e;
        if ((e = tmap_2d(&m.Xmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xc, H, rows, H * 2, 64, 64)) != FLP_OK) return e;
        if ((e = tmap_2d(&m.Dz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, dz_cols, dz_rows, dz_cols * 2, BK, BM)) != FLP_OK)
            return e;
        if ((e = tmap_2d(&m.DzMn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, dz_cols, dz_rows, dz_cols * 2, 64, 64)) != FLP_OK)
            return e;
        if ((e = tmap_2d(&m.DzSt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, dz_cols, dz_rows, dz_cols * 2, 32, BM,
                         CU_TENSOR_MAP_SWIZZLE_64B)) != FLP_OK)
            return e;
        if (dx_scratch)
            return tmap_2d(&m.Dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, scr + r0 * H, H, rows, H * 4, box_f32, BM,
                           out_swz);
        uint8_t* dXc = static_cast<uint8_t*>(dX) + r0 * H * dx_es;
        if (dX_dtype == FLP_F32)
            return tmap_2d(&m.Dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dXc, H, rows, H * 4, box_f32, BM, out_swz);
        return tmap_2d(&m.Dx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dXc, H, rows, H * 2, box_bf16, BM, out_swz);
    };

    std::vector<LaunchSpec> plan;
    if ((st = plan_backward_launches(M, H, V, ch, pairs, accumulate_dW, plan)) != FLP_OK) return st;

    BwdParams base{};
    base.V = static_cast<int>(V);
    base.KB_h = static_cast<int>(cdiv(H, BK));
    base.dx_f32 = (dX_dtype == FLP_F32 || dx_scratch) ? 1 : 0;
    base.dw_bf16 = dW_dtype == FLP_BF16;
    base.ent = ent;
    base.ignore_index = ignore_index;
    base.scale = scale;
    base.scale2 = scale * LOG2E;
    uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + L.off_cnt);
    base.row_dz = cnt;
    base.col_dz = cnt + L.Mt_max;
    base.dx_done = cnt + L.Mt_max + L.Vt;
    base.dw_done = cnt + 2 * L.Mt_max + L.Vt;
    base.ticket = reinterpret_cast<unsigned long long*>(ws + kTicketOffset);
    base.err = err;
    base.wait_limit_ns = kWaitLimitNs;
    // the fused schedule's tile counters start at zero and only grow
    if (ch.schedule == FLP_BWD_FUSED) FLP_CUDA(cudaMemsetAsync(ws + L.off_cnt, 0, L.cnt_bytes, s));

    int64_t mapped_r0 = -1, mapped_rows = -1;
    bool after_kernel = false;  // the first launch follows the header memset
    for (LaunchSpec& spec : plan) {
        NvtxRange launch_range("flp_backward_launch");
        if (spec.r0 != mapped_r0 || spec.rows != mapped_rows) {
            if ((st = row_maps(spec.r0, spec.rows, spec.dz_rows, spec.dz_cols)) != FLP_OK) return st;
            mapped_r0 = spec.r0;
            mapped_rows = spec.rows;
        }
        BwdParams& p = spec.p;
        const int64_t r0 = spec.r0;
        p.V = base.V;
        p.KB_h = base.KB_h;
        p.dx_f32 = base.dx_f32;
        p.dw_bf16 = base.dw_bf16;
        p.ent = base.ent;
        p.ignore_index = base.ignore_index;
        p.scale = base.scale;
        p.scale2 = base.scale2;
        p.y = reinterpret_cast<const long long*>(targets) + r0;
        p.lse = lse + r0;
        p.ent_v = ent ? entropy + r0 : nullptr;
        p.g_lp = grad_logprob ? grad_logprob + r0 : nullptr;
        p.g_ent = (ent && grad_entropy) ? grad_entropy + r0 : nullptr;
        p.row_dz = base.row_dz;
        p.col_dz = base.col_dz;
        p.dx_done = base.dx_done;
        p.dw_done = base.dw_done;
        p.ticket = base.ticket;
        p.ticket_base = ticket_base;
        p.err = base.err;
        p.wait_limit_ns = base.wait_limit_ns;
        if (spec.mark_begin >= 0) mark(spec.mark_begin, s);
        if ((st = launch_bwd(pairs, m, p, &ticket_base, s, after_kernel, narrow)) != FLP_OK) return st;
        if (spec.mark_end >= 0) mark(spec.mark_end, s);
        after_kernel = true;
    }
    if (dx_scratch) {
        const int64_t n = M * H;
        const int blocks = static_cast<int>(std::min<int64_t>(cdiv(n, 8 * 256), 8 * d->sm_count));
        flp_round_bf16_kernel<<<blocks, 256, 0, s>>>(scr, static_cast<uint16_t*>(dX), n);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "flp_round_bf16_kernel launch");
    }
    return FLP_OK;
}

flp_status flp_backward_schedule(int64_t M, int64_t H, int64_t V, size_t workspace_bytes,
                                 flp_bwd_schedule schedule, int pairs, int32_t* units,
                                 int64_t capacity, int64_t* count) {
    if (M < 0 || H < 1 || V < 1 || pairs < 1 || capacity < 0 || !count)
        return fail(FLP_ERR_INVALID_ARG, "M >= 0, H >= 1, V >= 1, pairs >= 1 and count required");
    BwdChoice ch{};
    flp_status st = choose_backward(M, H, V, workspace_bytes, schedule, &ch);
    if (st != FLP_OK) return st;
    std::vector<LaunchSpec> plan;
    if (M > 0 && (st = plan_backward_launches(M, H, V, ch, pairs, 0, plan)) != FLP_OK) return st;
    int64_t n = 0;
    for (size_t li = 0; li < plan.size(); ++li) {
        const BwdParams& p = plan[li].p;
        const int w0 = static_cast<int>(plan[li].r0 / std::max<int64_t>(1, ch.chunk));
        for (int u = 0; u < p.total; ++u, ++n) {
            if (!units || n >= capacity) continue;
            const BUnit t = decode_bwd(p, u);
            int32_t* e = units + 5 * n;
            e[0] = static_cast<int32_t>(li);
            // a wide dZ tile with its second half past the launch's vocabulary is listed as a dZ tile
            e[1] = !t.wide                 ? t.kind
                   : t.kind == kUnitDx     ? 3
                   : t.kind == kUnitDw     ? 5
                   : t.nt + 1 < p.vt_end   ? 4
                                           : kUnitDz;
            e[2] = t.wave + w0;  // split launches number their one wave 0
            e[3] = t.mt;
            e[4] = t.nt;
        }
    }
    *count = n;
    return FLP_OK;
}

flp_status flp_get_error(const void* workspace, void* stream) {
    if (!workspace) return fail(FLP_ERR_INVALID_ARG, "workspace must be non-null");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FLP_CUDA(cudaStreamSynchronize(s));
    int word = 0;
    FLP_CUDA(cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost));
    if (word & ERR_TIMEOUT) return FLP_ERR_TIMEOUT;
    if (word & ERR_BAD_TARGET) return FLP_ERR_BAD_TARGET;
    return FLP_OK;
}

}  // extern "C"

// ======================================================= allocation-free forward
//
// For callers that cannot allocate device memory (see flp_forward_noalloc in
// include/flp.h): the forward's scratch (header with the error word, the
// per-split partials and the target logits) lives in this file-scope device
// array instead of a caller workspace.  Host code only ever uses the array's
// device address, looked up once per device with that device current.

static __device__ __align__(256) uint8_t g_flp_static_scratch[FLP_STATIC_SCRATCH_BYTES];

namespace {

void* g_static_scratch_addr[kMaxDevices] = {};

flp_status static_scratch(int dev, uint8_t** out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_static_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_flp_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        if (!p) return fail(FLP_ERR_CUDA, "static scratch has no device address");
        g_static_scratch_addr[dev] = p;
    }
    *out = static_cast<uint8_t*>(g_static_scratch_addr[dev]);
    return FLP_OK;
}

}  // namespace

extern "C" flp_status flp_forward_noalloc(const void* X, const void* W, const int64_t* targets,
                                          int64_t M, int64_t H, int64_t V, int64_t ignore_index,
                                          float scale, int compute_entropy, float* logprob,
                                          float* lse, float* entropy, void* stream) {
    NvtxRange range("flp_forward_noalloc");
    const int ent = compute_entropy ? 1 : 0;
    flp_status st = forward_checks(X, W, targets, M, H, V, scale, ent, logprob, lse, entropy);
    if (st != FLP_OK) return st;
    DevInfo* d;
    int dev = 0;
    st = device_info(&d, &dev);
    if (st != FLP_OK) return st;
    st = check_device(&d);
    if (st != FLP_OK) return st;
    if (M > 0 && (st = check_on_current_device(X, "X")) != FLP_OK) return st;
    // the fastest split plan whose scratch fits the static array
    const FwdPlan f = plan_forward(M, H, V, ent, d->pairs, FLP_STATIC_SCRATCH_BYTES);
    if (f.bytes > FLP_STATIC_SCRATCH_BYTES) {
        char buf[200];
        snprintf(buf, sizeof buf,
                 "problem needs %zu bytes of forward scratch; the static scratch holds %u bytes",
                 f.bytes, static_cast<unsigned>(FLP_STATIC_SCRATCH_BYTES));
        return fail(FLP_ERR_UNSUPPORTED, buf);
    }
    uint8_t* ws = nullptr;
    st = static_scratch(dev, &ws);
    if (st != FLP_OK) return st;
    // the array keeps the last call's contents: launch_forward clears the header
    return launch_forward(X, W, targets, M, H, V, ignore_index, scale, ent, logprob, lse, entropy, f, ws,
                          kWaitLimitNs, -1, static_cast<cudaStream_t>(stream));
}

// ================================================ bounded-wait self-test

extern "C" flp_status flp_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                                int stall_after, int64_t wait_limit_ns,
                                                void* stream) {
    if (!workspace || !aligned16(workspace) || workspace_bytes < FLP_SELFTEST_WORKSPACE_BYTES)
        return fail(FLP_ERR_WORKSPACE, "self-test needs FLP_SELFTEST_WORKSPACE_BYTES of workspace");
    if (wait_limit_ns <= 0 || wait_limit_ns > 60ll * 1000 * 1000 * 1000)
        return fail(FLP_ERR_INVALID_ARG, "wait_limit_ns must be in (0, 60 s]");
    DevInfo* d;
    flp_status st = check_device(&d);
    if (st != FLP_OK) return st;
    constexpr int64_t M = 256, H = 256, V = 512;
    const FwdPlan f = plan_forward(M, H, V, 1, d->pairs);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t off_x = align_up(f.bytes, 1024);
    const size_t off_w = off_x + align_up(M * H * 2, 1024);
    const size_t off_y = off_w + align_up(V * H * 2, 1024);
    const size_t off_o = FLP_SELFTEST_OUTPUT_OFFSET;
    if (off_y + M * 8 > off_o || off_o + 3 * M * 4 > FLP_SELFTEST_WORKSPACE_BYTES)
        return fail(FLP_ERR_UNSUPPORTED, "self-test layout exceeds its workspace");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FLP_CUDA(cudaMemsetAsync(ws, 0, off_y + M * 8, s));  // header, inputs (zeros) and targets (0)
    float* out = reinterpret_cast<float*>(ws + off_o);   // logprob, lse, entropy: fp32 [M] each
    st = launch_forward(ws + off_x, ws + off_w, reinterpret_cast<const int64_t*>(ws + off_y), M, H, V, -100,
                        1.f, 1, out, out + M, out + 2 * M, f, ws, static_cast<unsigned long long>(wait_limit_ns),
                        stall_after < 0 ? -1 : stall_after, s);
    if (st != FLP_OK) return st;
    return flp_get_error(workspace, stream);
}

// A fused-schedule launch on a small internal all-zero problem (M = H = V =
// 256: one tile of each kind) laid out in the workspace.  broken != 0 drops
// the dZ tiles from the schedule, so the dX tile's dependency wait can never
// be met and has to give up after wait_limit_ns.
extern "C" flp_status flp_selftest_dependency_timeout(void* workspace, size_t workspace_bytes,
                                                      int broken, int64_t wait_limit_ns,
                                                      void* stream) {
    if (!workspace || !aligned16(workspace) || workspace_bytes < FLP_SELFTEST_WORKSPACE_BYTES)
        return fail(FLP_ERR_WORKSPACE, "self-test needs FLP_SELFTEST_WORKSPACE_BYTES of workspace");
    if (wait_limit_ns <= 0 || wait_limit_ns > 60ll * 1000 * 1000 * 1000)
        return fail(FLP_ERR_INVALID_ARG, "wait_limit_ns must be in (0, 60 s]");
    DevInfo* d;
    flp_status st = check_device(&d);
    if (st != FLP_OK) return st;
    constexpr int64_t M = 256, H = 256, V = 256;
    const BwdLayout L = bwd_layout(M, V);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t off_x = align_up(L.off_dz + M * L.Vp * 2, 1024);
    const size_t off_w = off_x + align_up(M * H * 2, 1024);
    const size_t off_y = off_w + align_up(V * H * 2, 1024);
    const size_t off_f = off_y + align_up(M * 8, 1024);  // lse, g_lp: fp32 [M] each
    const size_t off_dx = off_f + align_up(2 * M * 4, 1024);
    const size_t off_dw = off_dx + align_up(M * H * 2, 1024);
    const size_t end = off_dw + V * H * 4;
    if (end > FLP_SELFTEST_WORKSPACE_BYTES)
        return fail(FLP_ERR_UNSUPPORTED, "self-test layout exceeds its workspace");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FLP_CUDA(cudaMemsetAsync(ws, 0, end, s));  // header, counters, inputs (zeros), targets (0)

    BwdMaps m{};
    const void* X = ws + off_x;
    const void* W = ws + off_w;
    void* dz = ws + L.off_dz;
    if ((st = tmap_2d(&m.Xk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, H, M, H * 2, BK, BM)) != FLP_OK) return st;
    if ((st = tmap_2d(&m.Xmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, H, M, H * 2, 64, 64)) != FLP_OK) return st;
    if ((st = tmap_2d(&m.Wk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, BK, BNH)) != FLP_OK) return st;
    if ((st = tmap_2d(&m.Wmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, 64, 64)) != FLP_OK) return st;
    if ((st = tmap_2d(&m.Dz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, L.Vp, M, L.Vp * 2, BK, BM)) != FLP_OK) return st;
    if ((st = tmap_2d(&m.DzMn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, L.Vp, M, L.Vp * 2, 64, 64)) != FLP_OK) return st;
    if ((st = tmap_2d(&m.Dx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws + off_dx, H, M, H * 2, 64, BM)) != FLP_OK) return st;
    if ((st = tmap_2d(&m.Dw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ws + off_dw, H, V, H * 4, 32, BM)) != FLP_OK) return st;

    BwdChoice ch{FLP_BWD_FUSED, M, 1, L.Vp, 0, L.off_dz};
    std::vector<LaunchSpec> plan;
    if ((st = plan_backward_launches(M, H, V, ch, d->pairs, 0, plan)) != FLP_OK) return st;
    if (plan.size() != 1) return fail(FLP_ERR_UNSUPPORTED, "self-test schedule is not one launch");
    BwdParams& p = plan[0].p;
    if (broken) {
        p.nseg = 0;
        p.total = 0;
        SegList sl{&p};
        sl.add(kSegDx, 0, 0, 1, 0, 0, 1);  // the dX tile alone: its dZ tile never comes
    }
    uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + L.off_cnt);
    p.V = static_cast<int>(V);
    p.KB_h = static_cast<int>(H / BK);
    p.KB_v = static_cast<int>(L.Vp / BK);
    p.ignore_index = -100;
    p.scale = 1.f;
    p.scale2 = LOG2E;
    p.y = reinterpret_cast<const long long*>(ws + off_y);
    p.lse = reinterpret_cast<const float*>(ws + off_f);
    p.g_lp = reinterpret_cast<const float*>(ws + off_f + M * 4);
    p.row_dz = cnt;
    p.col_dz = cnt + L.Mt_max;
    p.dx_done = cnt + L.Mt_max + L.Vt;
    p.dw_done = cnt + 2 * L.Mt_max + L.Vt;
    p.ticket = reinterpret_cast<unsigned long long*>(ws + kTicketOffset);
    p.ticket_base = 0;
    p.err = reinterpret_cast<int*>(ws);
    p.wait_limit_ns = static_cast<unsigned long long>(wait_limit_ns);
    unsigned long long tb = 0;
    if ((st = launch_bwd(d->pairs, m, p, &tb, s)) != FLP_OK) return st;
    return flp_get_error(workspace, stream);
}

// The split schedule's dZ kernel (flp_dz_kernel) on a small internal all-zero
// problem (M = 256, H = 256, V = 512: one 256 x 512 tile) laid out in the
// workspace; stall_after >= 0 stops its producers after that many stages.
extern "C" flp_status flp_selftest_dz_wait_timeout(void* workspace, size_t workspace_bytes,
                                                   int stall_after, int64_t wait_limit_ns,
                                                   void* stream) {
    if (!workspace || !aligned16(workspace) || workspace_bytes < FLP_SELFTEST_WORKSPACE_BYTES)
        return fail(FLP_ERR_WORKSPACE, "self-test needs FLP_SELFTEST_WORKSPACE_BYTES of workspace");
    if (wait_limit_ns <= 0 || wait_limit_ns > 60ll * 1000 * 1000 * 1000)
        return fail(FLP_ERR_INVALID_ARG, "wait_limit_ns must be in (0, 60 s]");
    DevInfo* d;
    flp_status st = check_device(&d);
    if (st != FLP_OK) return st;
    constexpr int64_t M = 256, H = 256, V = 512;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t off_dz = kHeaderBytes;
    const size_t off_x = align_up(off_dz + M * V * 2, 1024);
    const size_t off_w = off_x + align_up(M * H * 2, 1024);
    const size_t off_y = off_w + align_up(V * H * 2, 1024);
    const size_t off_f = off_y + align_up(M * 8, 1024);  // lse, g_lp: fp32 [M] each
    const size_t end = off_f + 2 * M * 4;
    if (end > FLP_SELFTEST_WORKSPACE_BYTES)
        return fail(FLP_ERR_UNSUPPORTED, "self-test layout exceeds its workspace");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FLP_CUDA(cudaMemsetAsync(ws, 0, end, s));  // header, dZ, inputs (zeros), targets (0)

    BwdMaps m{};
    if ((st = tmap_2d(&m.Xk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws + off_x, H, M, H * 2, BK, BM)) != FLP_OK)
        return st;
    if ((st = tmap_2d(&m.Wk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws + off_w, H, V, H * 2, BK, BNH)) != FLP_OK)
        return st;
    if ((st = tmap_2d(&m.DzSt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws + off_dz, V, M, V * 2, 32, BM,
                      CU_TENSOR_MAP_SWIZZLE_64B)) != FLP_OK)
        return st;
    BwdParams p{};
    SegList sl{&p};
    sl.add(kSegDz2, 0, 0, 1, 0, 0, 1);  // the one wide dZ tile
    p.M = static_cast<int>(M);
    p.V = static_cast<int>(V);
    p.chunk = static_cast<int>(M);
    p.nwaves = 1;
    p.Mt_full = 1;
    p.Vt = static_cast<int>(V / BN);
    p.vt0 = 0;
    p.vt_end = p.Vt;
    p.KB_h = static_cast<int>(H / BK);
    p.static_order = 1;
    p.ignore_index = -100;
    p.scale = 1.f;
    p.scale2 = LOG2E;
    p.y = reinterpret_cast<const long long*>(ws + off_y);
    p.lse = reinterpret_cast<const float*>(ws + off_f);
    p.g_lp = reinterpret_cast<const float*>(ws + off_f + M * 4);
    p.err = reinterpret_cast<int*>(ws);
    p.wait_limit_ns = static_cast<unsigned long long>(wait_limit_ns);
    p.debug_stop_at = stall_after < 0 ? 0 : stall_after + 1;
    unsigned long long tb = 0;
    if ((st = launch_bwd(d->pairs, m, p, &tb, s)) != FLP_OK) return st;
    return flp_get_error(workspace, stream);
}

// ============================================================ loss heads

extern "C" flp_status flp_loss(const float* logprob, const int64_t* targets, int64_t M,
                               int64_t ignore_index, int kind, const float* old_logprob,
                               const float* advantage, const float* ref_logprob, float eps_low,
                               float eps_high, float beta, float* per_token_loss,
                               float* grad_logprob, float* loss, void* stream) {
    if (M < 0) return fail(FLP_ERR_INVALID_ARG, "M >= 0 required");
    if (kind != FLP_LOSS_NLL_MEAN && kind != FLP_LOSS_CLIPPED_SURROGATE && kind != FLP_LOSS_NLL_SUM)
        return fail(FLP_ERR_INVALID_ARG, "unknown loss kind");
    if (!loss || (M > 0 && (!logprob || !targets)))
        return fail(FLP_ERR_INVALID_ARG, "logprob, targets and loss must be non-null");
    if (kind == FLP_LOSS_CLIPPED_SURROGATE && M > 0 && (!old_logprob || !advantage))
        return fail(FLP_ERR_INVALID_ARG, "the clipped surrogate needs old_logprob and advantage");
    if (!(eps_low >= 0.f && eps_low <= 1.f && eps_high >= 0.f && std::isfinite(eps_high) &&
          std::isfinite(beta)))
        return fail(FLP_ERR_INVALID_ARG, "eps_low in [0, 1], eps_high >= 0 and beta finite required");
    DevInfo* d;
    flp_status st = device_info(&d, nullptr);
    if (st != FLP_OK) return st;
    LossParams p{};
    p.lp = logprob;
    p.y = reinterpret_cast<const long long*>(targets);
    p.M = M;
    p.ignore_index = ignore_index;
    p.kind = kind;
    p.old_lp = old_logprob;
    p.adv = advantage;
    p.ref_lp = ref_logprob;
    p.eps_low = eps_low;
    p.eps_high = eps_high;
    p.beta = beta;
    p.per_row = per_token_loss;
    p.grad = grad_logprob;
    p.loss = loss;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    flp_loss_kernel<<<1, LOSS_THREADS, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "flp_loss_kernel launch");
    return FLP_OK;
}

extern "C" flp_status flp_policy_loss(const float* logprob, const int64_t* targets, int64_t M,
                                      int64_t ignore_index, const int64_t* seq_offsets,
                                      int64_t num_seqs, const float* old_logprob,
                                      const float* advantage, const float* ref_logprob, float eps_low,
                                      float eps_high, float beta, int is_level, int aggregation,
                                      double normalizer, float* per_token_loss, float* grad_logprob,
                                      float* loss, void* stream) {
    if (M < 0) return fail(FLP_ERR_INVALID_ARG, "M >= 0 required");
    if (is_level != FLP_IS_TOKEN && is_level != FLP_IS_SEQUENCE)
        return fail(FLP_ERR_INVALID_ARG, "is_level must be FLP_IS_TOKEN or FLP_IS_SEQUENCE");
    if (aggregation != FLP_AGG_TOKEN_MEAN && aggregation != FLP_AGG_SEQUENCE_MEAN &&
        aggregation != FLP_AGG_SUM_OVER)
        return fail(FLP_ERR_INVALID_ARG, "unknown aggregation");
    if (!loss || (M > 0 && (!logprob || !targets || !old_logprob || !advantage)))
        return fail(FLP_ERR_INVALID_ARG, "logprob, targets, old_logprob, advantage and loss must be non-null");
    if (seq_offsets && num_seqs < 1)
        return fail(FLP_ERR_INVALID_ARG, "num_seqs >= 1 required with seq_offsets");
    if (!(eps_low >= 0.f && eps_low <= 1.f && eps_high >= 0.f && std::isfinite(eps_high) &&
          std::isfinite(beta) && std::isfinite(normalizer)))
        return fail(FLP_ERR_INVALID_ARG, "eps_low in [0, 1], eps_high >= 0, finite beta and normalizer required");
    DevInfo* d;
    flp_status st = device_info(&d, nullptr);
    if (st != FLP_OK) return st;
    PolicyLossParams p{};
    p.lp = logprob;
    p.y = reinterpret_cast<const long long*>(targets);
    p.M = M;
    p.ignore_index = ignore_index;
    p.off = reinterpret_cast<const long long*>(seq_offsets);
    p.B = seq_offsets ? num_seqs : 1;
    p.old_lp = old_logprob;
    p.adv = advantage;
    p.ref_lp = ref_logprob;
    p.eps_low = eps_low;
    p.eps_high = eps_high;
    p.beta = beta;
    p.is_level = is_level;
    p.aggregation = aggregation;
    p.normalizer = normalizer;
    p.per_row = per_token_loss;
    p.grad = grad_logprob;
    p.loss = loss;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    flp_policy_loss_kernel<<<1, LOSS_THREADS, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "flp_policy_loss_kernel launch");
    return FLP_OK;
}
