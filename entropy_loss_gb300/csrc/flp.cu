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

#include <nvtx3/nvToolsExt.h>

#include "flp.h"
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
                   uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    flp_status st = get_encode(&enc);
    if (st != FLP_OK) return st;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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

// Chooses the V-split: units are (256-row pair tile, run of tps 256-column
// tiles); a static round-robin over the persistent CTA pairs finishes after
// ceil(units / pairs) * tps tiles.  Each extra split adds M * 24 bytes of
// partial traffic, charged in tile-times so that near-ties favour fewer splits.
FwdPlan plan_forward(int64_t M, int64_t H, int64_t V, int compute_entropy, int pairs) {
    FwdPlan f{};
    pairs = std::max(1, pairs);
    f.Mt = static_cast<int>(cdiv(M, PM));
    f.Vt = static_cast<int>(cdiv(V, BN));
    const double tile_s = 2.0 * PM * BN * static_cast<double>(H) / 2.4e13;  // ~bf16 rate of a pair
    const double split_cost = (static_cast<double>(M) * 24.0 / 6.0e12) / tile_s;
    double best = 1e300;
    int best_tps = f.Vt;
    for (int tps = 1; tps <= f.Vt; ++tps) {
        const int S = static_cast<int>(cdiv(f.Vt, tps));
        if (tps > 1 && cdiv(f.Vt, tps - 1) == S) continue;  // same split count, shorter runs win
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
    const size_t part = align_up(static_cast<size_t>(f.S) * M * sizeof(float), 1024);
    f.off_m = kHeaderBytes;
    f.off_s = f.off_m + part;
    f.off_t = f.off_s + part;
    f.off_zy = f.off_t + (compute_entropy ? part : 0);
    f.bytes = f.off_zy + align_up(static_cast<size_t>(M) * sizeof(float), 1024);
    return f;
}

struct BwdPlan {
    int64_t Vp, chunk;
    size_t off_dz, bytes;
};

BwdPlan plan_backward(int64_t M, int64_t V, int64_t chunk_rows) {
    BwdPlan b{};
    b.Vp = cdiv(V, BN) * BN;
    const int64_t mr = std::max<int64_t>(BM, cdiv(M, BM) * BM);
    int64_t c = chunk_rows > 0 ? chunk_rows : kDefaultChunkRows;
    c = std::max<int64_t>(BM, cdiv(c, BM) * BM);
    b.chunk = std::min(c, mr);
    b.off_dz = kHeaderBytes;
    b.bytes = b.off_dz + static_cast<size_t>(b.chunk) * b.Vp * 2;
    return b;
}

bool smem_attrs_done(DevInfo* d) { return d->attrs_set; }

template <int kMode, bool kEnt>
cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(flp_tile_kernel<kMode, kEnt>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
}

template <bool kDxF32, bool kDwBf16>
cudaError_t set_bwd_smem_attr() {
    return cudaFuncSetAttribute(flp_bwd_gemm_kernel<kDxF32, kDwBf16>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
}

flp_status ensure_attrs(DevInfo* d) {
    if (smem_attrs_done(d)) return FLP_OK;
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = set_smem_attr<kFwd, true>();
    if (e == cudaSuccess) e = set_smem_attr<kFwd, false>();
    if (e == cudaSuccess) e = set_smem_attr<kDz, true>();
    if (e == cudaSuccess) e = set_smem_attr<kDz, false>();
    if (e == cudaSuccess) e = set_bwd_smem_attr<false, false>();
    if (e == cudaSuccess) e = set_bwd_smem_attr<true, false>();
    if (e == cudaSuccess) e = set_bwd_smem_attr<false, true>();
    if (e == cudaSuccess) e = set_bwd_smem_attr<true, true>();
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
    e = cudaOccupancyMaxActiveClusters(&clusters, flp_tile_kernel<kFwd, true>, &cfg);
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
// that share each tcgen05.mma.cta_group::2 tile).
template <typename... KArgs, typename... Args>
flp_status launch_pairs(void (*kernel)(KArgs...), int grid, cudaStream_t s, const char* what,
                        Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, what);
    return FLP_OK;
}

template <int kMode, bool kEnt>
flp_status launch_tile(int grid, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                       const TileParams& p, cudaStream_t s) {
    return launch_pairs(flp_tile_kernel<kMode, kEnt>, grid, s, "flp_tile_kernel launch", a, b, o, p);
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
                               int64_t chunk_rows, size_t* fwd_bytes, size_t* bwd_bytes) {
    if (M < 0 || H < 1 || V < 1) return fail(FLP_ERR_INVALID_ARG, "M >= 0, H >= 1 and V >= 1 required");
    DevInfo* d;
    flp_status st = check_device(&d);
    if (st != FLP_OK) return st;
    if (fwd_bytes) *fwd_bytes = plan_forward(M, H, V, compute_entropy ? 1 : 0, d->pairs).bytes;
    if (bwd_bytes) *bwd_bytes = plan_backward(M, V, chunk_rows).bytes;
    return FLP_OK;
}

flp_status flp_forward(const void* X, const void* W, const int64_t* targets, int64_t M,
                       int64_t H, int64_t V, int64_t ignore_index, float scale,
                       int compute_entropy, float* logprob, float* lse, float* entropy,
                       void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange range("flp_forward");
    flp_status st = common_checks(X, W, targets, M, H, V);
    if (st != FLP_OK) return st;
    const int ent = compute_entropy ? 1 : 0;
    if (M > 0 && (!logprob || !lse || (ent && !entropy) || (!ent && entropy)))
        return fail(FLP_ERR_INVALID_ARG, "logprob and lse required; entropy iff compute_entropy");
    if (!aligned16(logprob) || !aligned16(lse) || (entropy && !aligned16(entropy)))
        return fail(FLP_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(FLP_ERR_INVALID_ARG, "scale must be finite");
    DevInfo* d;
    st = check_device(&d);
    if (st != FLP_OK) return st;
    if (M > 0 && (st = check_on_current_device(X, "X")) != FLP_OK) return st;
    const FwdPlan f = plan_forward(M, H, V, ent, d->pairs);
    if (!workspace || workspace_bytes < f.bytes || !aligned16(workspace))
        return fail(FLP_ERR_WORKSPACE, "forward workspace null, misaligned or too small");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* err = reinterpret_cast<int*>(ws);
    FLP_CUDA(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
    if (M == 0) return FLP_OK;

    CUtensorMap tmX, tmW;
    st = tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, H, M, H * 2, BK, BM);
    if (st != FLP_OK) return st;
    st = tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, BK, BNH);
    if (st != FLP_OK) return st;

    TileParams p{};
    p.units = f.units;
    p.Mt = f.Mt;
    p.Nt = f.Vt;
    p.S = f.S;
    p.tps = f.tps;
    p.GM = f.GM;
    p.KB = static_cast<int>(cdiv(H, BK));
    p.M = static_cast<int>(M);
    p.V = static_cast<int>(V);
    p.row0 = 0;
    p.ignore_index = ignore_index;
    p.scale = scale;
    p.scale2 = scale * LOG2E;
    p.y = reinterpret_cast<const long long*>(targets);
    p.part_m = reinterpret_cast<float*>(ws + f.off_m);
    p.part_s = reinterpret_cast<float*>(ws + f.off_s);
    p.part_t = ent ? reinterpret_cast<float*>(ws + f.off_t) : nullptr;
    p.zy = reinterpret_cast<float*>(ws + f.off_zy);
    p.err = err;
    p.wait_limit_ns = kWaitLimitNs;
    p.debug_stall_after = -1;
    mark(0, s);
    st = ent ? launch_tile<kFwd, true>(f.grid, tmX, tmW, tmX, p, s)
             : launch_tile<kFwd, false>(f.grid, tmX, tmW, tmX, p, s);
    if (st != FLP_OK) return st;
    mark(1, s);

    MergeParams mp{};
    mp.M = static_cast<int>(M);
    mp.S = f.S;
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
    flp_merge_kernel<<<static_cast<unsigned>(cdiv(M, MERGE_ROWS)), MERGE_ROWS * MERGE_WAYS, 0, s>>>(mp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "flp_merge_kernel launch");
    mark(3, s);
    return FLP_OK;
}

flp_status flp_backward(const void* X, const void* W, const int64_t* targets, int64_t M,
                        int64_t H, int64_t V, int64_t ignore_index, float scale,
                        int compute_entropy, const float* lse, const float* entropy,
                        const float* grad_logprob, const float* grad_entropy, void* dX,
                        flp_dtype dX_dtype, void* dW, flp_dtype dW_dtype, int accumulate_dW,
                        void* workspace, size_t workspace_bytes, void* stream) {
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
    if (!workspace || !aligned16(workspace) || workspace_bytes < kHeaderBytes)
        return fail(FLP_ERR_WORKSPACE, "backward workspace null, misaligned or too small");
    // Largest wave (multiple of 128 rows, at most M rounded up) the workspace holds.
    const int64_t Vp = cdiv(V, BN) * BN;
    const int64_t fit = static_cast<int64_t>((workspace_bytes - kHeaderBytes) / (static_cast<size_t>(Vp) * 2));
    const int64_t mr = std::max<int64_t>(BM, cdiv(M, BM) * BM);
    const int64_t chunk = std::min(mr, fit / BM * BM);
    if (chunk < BM) return fail(FLP_ERR_WORKSPACE, "backward workspace holds fewer than 128 rows of dZ");
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
    void* dz = ws + kHeaderBytes;
    unsigned long long ticket_base = 0;

    CUtensorMap tmW_k, tmW_mn, tmDW;
    st = tmap_2d(&tmW_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, BK, BNH);
    if (st != FLP_OK) return st;
    st = tmap_2d(&tmW_mn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, 64, 64);
    if (st != FLP_OK) return st;
    if (dW_dtype == FLP_BF16)
        st = tmap_2d(&tmDW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dW, H, V, H * 2, 64, BM);
    else
        st = tmap_2d(&tmDW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dW, H, V, H * 4, 32, BM);
    if (st != FLP_OK) return st;

    const int Vt = static_cast<int>(Vp / BN);
    const int Nt_h = static_cast<int>(cdiv(H, BN));
    const int pairs = d->pairs;
    const int64_t gm_rows = std::max<int64_t>(4, 40ll * 1000 * 1000 / (PM * 2 * H));

    for (int64_t r0 = 0; r0 < M; r0 += chunk) {
        NvtxRange wave_range("flp_backward_wave");
        const int64_t rows = std::min(chunk, M - r0);
        const uint8_t* Xc = static_cast<const uint8_t*>(X) + r0 * H * 2;
        uint8_t* dXc = static_cast<uint8_t*>(dX) + r0 * H * dx_es;
        CUtensorMap tmXk, tmXmn, tmDZk, tmDZmn, tmDZst, tmDX;
        if ((st = tmap_2d(&tmXk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xc, H, rows, H * 2, BK, BM)) != FLP_OK) return st;
        if ((st = tmap_2d(&tmXmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xc, H, rows, H * 2, 64, 64)) != FLP_OK) return st;
        if ((st = tmap_2d(&tmDZst, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, Vp, rows, Vp * 2, 64, BM)) != FLP_OK) return st;
        if ((st = tmap_2d(&tmDZk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, Vp, rows, Vp * 2, BK, BM)) != FLP_OK) return st;
        if ((st = tmap_2d(&tmDZmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dz, Vp, rows, Vp * 2, 64, 64)) != FLP_OK) return st;
        if (dX_dtype == FLP_F32)
            st = tmap_2d(&tmDX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dXc, H, rows, H * 4, 32, BM);
        else
            st = tmap_2d(&tmDX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dXc, H, rows, H * 2, 64, BM);
        if (st != FLP_OK) return st;

        // (1) recompute logits tiles -> bf16 dZ for this wave
        TileParams p{};
        p.Mt = static_cast<int>(cdiv(rows, PM));
        p.Nt = Vt;
        p.S = Vt;
        p.tps = 1;
        p.GM = static_cast<int>(std::min<int64_t>(p.Mt, gm_rows));
        p.units = p.Mt * p.Nt;
        p.KB = static_cast<int>(cdiv(H, BK));
        p.M = static_cast<int>(rows);
        p.V = static_cast<int>(V);
        p.row0 = static_cast<int>(r0);
        p.ignore_index = ignore_index;
        p.scale = scale;
        p.scale2 = scale * LOG2E;
            p.y = reinterpret_cast<const long long*>(targets);
        p.lse = lse;
        p.ent = ent ? entropy : nullptr;
        p.g_lp = grad_logprob;
        p.g_ent = ent ? grad_entropy : nullptr;
        p.err = err;
        p.wait_limit_ns = kWaitLimitNs;
        p.debug_stall_after = -1;
        const int grid_dz = 2 * std::min(p.units, pairs);
        const bool first = (r0 == 0);
        if (first) mark(4, s);
        st = ent ? launch_tile<kDz, true>(grid_dz, tmXk, tmW_k, tmDZst, p, s)
                 : launch_tile<kDz, false>(grid_dz, tmXk, tmW_k, tmDZst, p, s);
        if (st != FLP_OK) return st;
        if (first) mark(5, s);

        // (2) dX[wave] = dZ W (K = Vp) and dW (+)= dZ^T X[wave] (K = wave rows),
        // one persistent launch of CTA pairs; the ticket counter lives in the
        // zeroed header and every launch consumes units + pairs tickets.
        BwdParams q{};
        q.Mt_dx = static_cast<int>(cdiv(rows, PM));
        q.GM_dx = std::min(q.Mt_dx, 8);
        q.Nt = Nt_h;
        q.units_dx = q.Mt_dx * Nt_h;
        q.units_dw = Vt * Nt_h;
        q.KB_dx = static_cast<int>(Vp / BK);
        q.KB_dw = static_cast<int>(cdiv(rows, BK));
        q.dw_add = (accumulate_dW || r0 > 0) ? 1 : 0;
        q.ticket = reinterpret_cast<unsigned long long*>(ws + kTicketOffset);
        q.ticket_base = ticket_base;
        q.err = err;
        q.wait_limit_ns = kWaitLimitNs;
        const int total = q.units_dx + q.units_dw;
        const int pairs_bw = std::min(total, pairs);
        ticket_base += static_cast<unsigned long long>(total) + pairs_bw;
        if (first) mark(6, s);
        const char* what = "flp_bwd_gemm_kernel launch";
        const int g = 2 * pairs_bw;
        if (dX_dtype == FLP_F32)
            st = (dW_dtype == FLP_BF16)
                     ? launch_pairs(flp_bwd_gemm_kernel<true, true>, g, s, what, tmDZk, tmW_mn, tmDZmn, tmXmn, tmDX, tmDW, q)
                     : launch_pairs(flp_bwd_gemm_kernel<true, false>, g, s, what, tmDZk, tmW_mn, tmDZmn, tmXmn, tmDX, tmDW, q);
        else
            st = (dW_dtype == FLP_BF16)
                     ? launch_pairs(flp_bwd_gemm_kernel<false, true>, g, s, what, tmDZk, tmW_mn, tmDZmn, tmXmn, tmDX, tmDW, q)
                     : launch_pairs(flp_bwd_gemm_kernel<false, false>, g, s, what, tmDZk, tmW_mn, tmDZmn, tmXmn, tmDX, tmDW, q);
        if (st != FLP_OK) return st;
        if (first) mark(7, s);
    }
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
    flp_status st = common_checks(X, W, targets, M, H, V);
    if (st != FLP_OK) return st;
    const int ent = compute_entropy ? 1 : 0;
    if (M > 0 && (!logprob || !lse || (ent && !entropy) || (!ent && entropy)))
        return fail(FLP_ERR_INVALID_ARG, "logprob and lse required; entropy iff compute_entropy");
    if (!aligned16(logprob) || !aligned16(lse) || (entropy && !aligned16(entropy)))
        return fail(FLP_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(FLP_ERR_INVALID_ARG, "scale must be finite");
    DevInfo* d;
    int dev = 0;
    st = device_info(&d, &dev);
    if (st != FLP_OK) return st;
    st = check_device(&d);
    if (st != FLP_OK) return st;
    if (M > 0 && (st = check_on_current_device(X, "X")) != FLP_OK) return st;
    const FwdPlan f = plan_forward(M, H, V, ent, d->pairs);
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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = reinterpret_cast<int*>(ws);
    FLP_CUDA(cudaMemsetAsync(ws, 0, kHeaderBytes, s));  // the array keeps the last call's contents
    if (M == 0) return FLP_OK;

    CUtensorMap tmX, tmW;
    st = tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, H, M, H * 2, BK, BM);
    if (st != FLP_OK) return st;
    st = tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, H, V, H * 2, BK, BNH);
    if (st != FLP_OK) return st;

    TileParams p{};
    p.units = f.units;
    p.Mt = f.Mt;
    p.Nt = f.Vt;
    p.S = f.S;
    p.tps = f.tps;
    p.GM = f.GM;
    p.KB = static_cast<int>(cdiv(H, BK));
    p.M = static_cast<int>(M);
    p.V = static_cast<int>(V);
    p.row0 = 0;
    p.ignore_index = ignore_index;
    p.scale = scale;
    p.scale2 = scale * LOG2E;
    p.y = reinterpret_cast<const long long*>(targets);
    p.part_m = reinterpret_cast<float*>(ws + f.off_m);
    p.part_s = reinterpret_cast<float*>(ws + f.off_s);
    p.part_t = ent ? reinterpret_cast<float*>(ws + f.off_t) : nullptr;
    p.zy = reinterpret_cast<float*>(ws + f.off_zy);
    p.err = err;
    p.wait_limit_ns = kWaitLimitNs;
    p.debug_stall_after = -1;
    st = ent ? launch_tile<kFwd, true>(f.grid, tmX, tmW, tmX, p, s)
             : launch_tile<kFwd, false>(f.grid, tmX, tmW, tmX, p, s);
    if (st != FLP_OK) return st;

    MergeParams mp{};
    mp.M = static_cast<int>(M);
    mp.S = f.S;
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
    flp_merge_kernel<<<static_cast<unsigned>(cdiv(M, MERGE_ROWS)), MERGE_ROWS * MERGE_WAYS, 0, s>>>(mp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "flp_merge_kernel launch");
    return FLP_OK;
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
    if (off_y + M * 8 > FLP_SELFTEST_WORKSPACE_BYTES)
        return fail(FLP_ERR_UNSUPPORTED, "self-test layout exceeds its workspace");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FLP_CUDA(cudaMemsetAsync(ws, 0, off_y + M * 8, s));  // header, inputs (zeros) and targets (0)

    CUtensorMap tmX, tmW;
    st = tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws + off_x, H, M, H * 2, BK, BM);
    if (st != FLP_OK) return st;
    st = tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws + off_w, H, V, H * 2, BK, BNH);
    if (st != FLP_OK) return st;
    TileParams p{};
    p.units = f.units;
    p.Mt = f.Mt;
    p.Nt = f.Vt;
    p.S = f.S;
    p.tps = f.tps;
    p.GM = f.GM;
    p.KB = static_cast<int>(cdiv(H, BK));
    p.M = static_cast<int>(M);
    p.V = static_cast<int>(V);
    p.ignore_index = -100;
    p.scale = 1.f;
    p.scale2 = LOG2E;
    p.y = reinterpret_cast<const long long*>(ws + off_y);
    p.part_m = reinterpret_cast<float*>(ws + f.off_m);
    p.part_s = reinterpret_cast<float*>(ws + f.off_s);
    p.part_t = reinterpret_cast<float*>(ws + f.off_t);
    p.zy = reinterpret_cast<float*>(ws + f.off_zy);
    p.err = reinterpret_cast<int*>(ws);
    p.wait_limit_ns = static_cast<unsigned long long>(wait_limit_ns);
    p.debug_stall_after = stall_after < 0 ? -1 : stall_after;
    st = launch_tile<kFwd, true>(f.grid, tmX, tmW, tmX, p, s);
    if (st != FLP_OK) return st;
    return flp_get_error(workspace, stream);
}

// ============================================================ loss heads

extern "C" flp_status flp_loss(const float* logprob, const int64_t* targets, int64_t M,
                               int64_t ignore_index, int kind, const float* old_logprob,
                               const float* advantage, const float* ref_logprob, float eps_low,
                               float eps_high, float beta, float* per_token_loss,
                               float* grad_logprob, float* loss, void* stream) {
    if (M < 0) return fail(FLP_ERR_INVALID_ARG, "M >= 0 required");
    if (kind != FLP_LOSS_NLL_MEAN && kind != FLP_LOSS_CLIPPED_SURROGATE)
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
