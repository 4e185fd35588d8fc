// kernels.cuh - sm_103a kernels of the fused linear log-prob / cross-entropy head.
//
// Every contraction of the path runs on CTA pairs (clusters of two CTAs on two
// SMs) that share one 256 x 256 output tile: tcgen05.mma.cta_group::2 with
// M = 256 (128 rows of A in each CTA) and N = 256 (B split along N, 128 rows
// in each CTA), fp32 accumulators in both CTAs' TMEM.  Each SM therefore loads
// 16 KiB of A and 16 KiB of B per 64-deep K step for 2 * 128 * 256 * 64 MACs.
//
//   flp_tile_kernel<kFwd> : z = s X W^T tiles -> online max / sum-exp /
//                           (entropy) / target pick per row -> raw per-split
//                           partials (forward, fused epilogue)
//   flp_tile_kernel<kDz>  : z tiles recomputed -> dZ = s[g_lp(onehot - p) +
//                           g_ent p(sum pz - z)] in bf16, TMA-stored to the
//                           wave's dZ buffer
//   flp_bwd_gemm_kernel   : dX[wave] = dZ W and dW (+)= dZ^T X[wave] in one
//                           persistent launch with a ticket-counter scheduler
//
// Roles (192 threads per CTA, one CTA per SM):
//   warp 0      TMA producer (one lane) for this CTA's halves of A and B
//   warp 1      TMEM allocation (both CTAs) and, in the leader CTA (cluster
//               rank 0), the single thread that issues the pair MMAs
//   warps 2..5  epilogue: thread == accumulator row (TMEM lane) of this CTA
// Barriers: both CTAs' TMA loads complete on the leader's `full` barrier; the
// leader's MMA commits are multicast to both CTAs' `empty` (stage free) and
// `tfull` (accumulator ready) barriers; both CTAs' epilogues release an
// accumulator on the leader's `tempty` barrier.  Two 256-column accumulators
// (512 TMEM columns) let a tile's epilogue overlap the next tile's MMAs.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel raises the
// timeout bit in the error word, stops issuing work, lets its copies and MMAs
// in flight finish (a bounded wait), frees its TMEM and returns.
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"

namespace flp {

constexpr int BM = 128;           // rows of A per CTA (TMEM lanes)
constexpr int PM = 256;           // rows of the pair tile (UMMA M)
constexpr int BN = 256;           // columns of the pair tile (UMMA N)
constexpr int BNH = BN / 2;       // rows of B held by each CTA of the pair
constexpr int BK = 64;            // K per pipeline stage (one 128-byte swizzle atom)
constexpr int UMMA_K = 16;        // K per tcgen05.mma (bf16)
constexpr int STAGES = 6;
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint16_t PAIR_MASK = 0x3;

constexpr uint32_t A_STAGE_BYTES = BM * BK * 2;    // 16 KiB
constexpr uint32_t B_STAGE_BYTES = BNH * BK * 2;   // 16 KiB
constexpr uint32_t PAIR_STAGE_TX = 2 * (A_STAGE_BYTES + B_STAGE_BYTES);  // lands on the leader's barrier
constexpr uint32_t STG_BYTES = 128 * 128;          // one 128-row x 128-byte store box
constexpr uint32_t NUM_STG = 2;
constexpr int SCHED_SLOTS = 4;

constexpr int ERR_BAD_TARGET = 1;
constexpr int ERR_TIMEOUT = 2;

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

enum Mode : int { kFwd = 0, kDz = 1 };

// Offsets inside the (1024-byte aligned) dynamic shared memory block; the
// layout is identical in both CTAs of a pair, which the pair MMA relies on.
constexpr uint32_t SMEM_A = 0;
constexpr uint32_t SMEM_B = SMEM_A + STAGES * A_STAGE_BYTES;
constexpr uint32_t SMEM_STG = SMEM_B + STAGES * B_STAGE_BYTES;
constexpr uint32_t SMEM_BAR = SMEM_STG + NUM_STG * STG_BYTES;
// full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, sched_full[4], sched_empty[4]
constexpr uint32_t NUM_BARS = 2 * STAGES + 4 + 1 + 2 * SCHED_SLOTS;
constexpr uint32_t SMEM_MISC = SMEM_BAR + NUM_BARS * 8;  // tmem slot, abort flag, sched slots
constexpr uint32_t SMEM_TOTAL = SMEM_MISC + 8 + 4 * SCHED_SLOTS;
constexpr uint32_t SMEM_ALLOC = SMEM_TOTAL + 1024;  // slack for 1024-byte alignment

struct Smem {
    uint8_t* base;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint64_t* sched_full;
    uint64_t* sched_empty;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    volatile int* sched_val;
};

__device__ __forceinline__ Smem smem_layout(uint8_t* raw) {
    Smem s;
    s.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.base + SMEM_BAR);
    s.full = bars;
    s.empty = bars + STAGES;
    s.tfull = bars + 2 * STAGES;
    s.tempty = bars + 2 * STAGES + 2;
    s.drain = bars + 2 * STAGES + 4;
    s.sched_full = bars + 2 * STAGES + 5;
    s.sched_empty = s.sched_full + SCHED_SLOTS;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.base + SMEM_MISC);
    s.abort_flag = reinterpret_cast<volatile int*>(s.base + SMEM_MISC + 4);
    s.sched_val = reinterpret_cast<volatile int*>(s.base + SMEM_MISC + 8);
    return s;
}

// Records a timeout in the error word and tells both CTAs of the pair to stop
// waiting (the peer's flag is written through the cluster window).
__device__ __forceinline__ void raise_abort(const Smem& sm, int* err) {
    atomicOr(err, ERR_TIMEOUT);
    *sm.abort_flag = 1;
    const uint32_t peer = cluster_ctarank() ^ 1u;
    st_shared_cluster_u32(mapa_shared(smem_addr(const_cast<int*>(sm.abort_flag)), peer), 1u);
}

// Barrier set-up, TMEM allocation on both CTAs, and the cluster handshake that
// makes the peer's barriers visible before any remote arrive or TMA signal.
__device__ __forceinline__ uint32_t pair_prologue(const Smem& sm, int warp) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm.tfull[a], 1);
            mbar_init(&sm.tempty[a], 2 * EPI_THREADS);
        }
        mbar_init(sm.drain, 1);
        for (int s = 0; s < SCHED_SLOTS; ++s) {
            mbar_init(&sm.sched_full[s], 1);
            mbar_init(&sm.sched_empty[s], 2 + 2 * EPI_THREADS);
        }
        *sm.abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(sm.tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    return *sm.tmem_slot;
}

// Teardown: on an abort give copies in flight a bounded grace period, then a
// cluster handshake (no CTA leaves while its peer may still touch its shared
// memory or TMEM) and the pair TMEM release.
__device__ __forceinline__ void pair_epilogue(const Smem& sm, int warp, uint32_t tmem_base) {
    if (*sm.abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// Operand descriptors for UMMA step k (0..3) inside a 64-deep stage.
template <int kMN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int k) {
    if constexpr (kMN == 0)
        return sdesc_sw128(base + k * (UMMA_K * 2), 16, 1024);  // K-major: 32 B inside the atom
    else
        return sdesc_sw128(base + k * (UMMA_K * 128), 8192, 1024);  // MN-major: 16 rows of 128 B
}

// ------------------------------------------------------------ epilogue pieces

// v[idx] for a thread-dependent idx in [0, 32) through a 5-level select tree,
// so the 32 values stay in registers (no dynamically indexed local array).
__device__ __forceinline__ float select32(const uint32_t (&v)[32], int idx) {
    uint32_t a[16], b[8], c[4], d[2];
#pragma unroll
    for (int j = 0; j < 16; ++j) a[j] = (idx & 16) ? v[j + 16] : v[j];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = (idx & 8) ? a[j + 8] : a[j];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = (idx & 4) ? b[j + 4] : b[j];
#pragma unroll
    for (int j = 0; j < 2; ++j) d[j] = (idx & 2) ? c[j + 2] : c[j];
    return __uint_as_float((idx & 1) ? d[1] : d[0]);
}

// Write 8 x 16-byte chunks of one row into a 128B-swizzled 128-row box.
__device__ __forceinline__ void stage_row(uint32_t box_base, int r, const uint32_t (&w)[32]) {
    const uint32_t row_addr = box_base + r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        st_shared_v4(row_addr + ((c ^ (r & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                     w[4 * c + 3]);
}

// Two store boxes used in turn: before a box is rewritten, the bulk store
// that last read it must have finished reading.
struct StoreRing {
    uint32_t n = 0;
};

__device__ __forceinline__ uint32_t store_box_acquire(StoreRing& ring, uint8_t* smem, int et) {
    const uint32_t buf = ring.n & 1u;
    if (ring.n >= NUM_STG) {
        if (et == 0) bulk_wait_group_read<NUM_STG - 1>();
        named_bar_sync(1, EPI_THREADS);
    }
    return smem_addr(smem + SMEM_STG + buf * STG_BYTES);
}

__device__ __forceinline__ void store_box_release(StoreRing& ring, uint8_t* smem, int et,
                                                  const CUtensorMap* tmOut, int x, int y, bool add) {
    const uint32_t buf = ring.n & 1u;
    fence_proxy_async_smem();
    named_bar_sync(1, EPI_THREADS);
    if (et == 0) {
        const void* src = smem + SMEM_STG + buf * STG_BYTES;
        if (add)
            tma_reduce_add_2d(tmOut, src, x, y);
        else
            tma_store_2d(tmOut, src, x, y);
        bulk_commit_group();
    }
    ring.n++;
}

// fp32 accumulator columns [c0, c0 + 64) of this thread's row -> 32 packed bf16 pairs.
__device__ __forceinline__ void tmem_row64_to_bf16(uint32_t taddr, uint32_t (&w)[32]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + h * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
            w[h * 16 + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
    }
}

// ------------------------------------------------------- forward / dZ kernel

struct TileParams {
    // schedule: units are runs [n0, n1) of 256-column tiles sharing one 256-row pair tile
    int units, Mt, Nt, S, tps, GM;
    int KB;    // K blocks of 64 (H / 64, rounded up)
    int M;     // rows of this launch (all rows for kFwd, the wave's rows for kDz)
    int V;     // vocabulary size (column mask)
    int row0;  // first global row of the wave (kDz)
    long long ignore_index;
    float scale;   // s
    float scale2;  // s * log2(e)
    const long long* y;
    const float* lse;
    const float* ent;
    const float* g_lp;
    const float* g_ent;
    float* part_m;
    float* part_s;
    float* part_t;
    float* zy;
    int* err;
    unsigned long long wait_limit_ns;
    int debug_stall_after;  // < 0: off; else the producers stop after this many stages
};

struct Unit {
    int mt, n0, n1, split;
};

// Units are ordered in groups of GM pair M-tiles; inside a group the split index
// is outermost, so the pairs running at the same time share W tiles while the
// group's X rows stay resident in L2.
__device__ __forceinline__ Unit decode_unit(const TileParams& p, int u) {
    const int per_group = p.GM * p.S;
    const int g = u / per_group;
    const int first_m = g * p.GM;
    const int gm = min(p.GM, p.Mt - first_m);
    const int r = u - g * per_group;
    Unit t;
    t.split = r / gm;
    t.mt = first_m + (r - t.split * gm);
    t.n0 = t.split * p.tps;
    t.n1 = min(p.Nt, t.n0 + p.tps);
    return t;
}

template <int kMode, bool kEnt>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    flp_tile_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmOut, const TileParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = smem_layout(smem_raw);
    uint8_t* smem = sm.base;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if constexpr (kMode == kDz) tma_prefetch_desc(&tmOut);
    }
    const uint32_t tmem_base = pair_prologue(sm, warp);
    const uint64_t limit = p.wait_limit_ns;
    volatile int* abort_flag = sm.abort_flag;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int u = pair; u < p.units && ok; u += npairs) {
                const Unit t = decode_unit(p, u);
                for (int nt = t.n0; nt < t.n1 && ok; ++nt) {
                    for (int kb = 0; kb < p.KB; ++kb) {
                        if (p.debug_stall_after >= 0 && issued >= p.debug_stall_after) {
                            ok = false;  // injected stall: stop feeding the MMA
                            break;
                        }
                        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, limit, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(&sm.full[stage], PAIR_STAGE_TX);
                        const uint32_t bar = mapa_shared(smem_addr(&sm.full[stage]), 0);
                        tma_load_2d_pair(smem + SMEM_A + stage * A_STAGE_BYTES, &tmA, kb * BK,
                                         t.mt * PM + static_cast<int>(rank) * BM, bar);
                        tma_load_2d_pair(smem + SMEM_B + stage * B_STAGE_BYTES, &tmB, kb * BK,
                                         nt * BN + static_cast<int>(rank) * BNH, bar);
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (!ok && p.debug_stall_after < 0) {
                raise_abort(sm, p.err);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------- MMA issuer (leader)
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            constexpr uint32_t idesc = idesc_bf16_f32(PM, BN, 0, 0);
            for (int u = pair; u < p.units && ok; u += npairs) {
                const Unit t = decode_unit(p, u);
                for (int nt = t.n0; nt < t.n1 && ok; ++nt) {
                    if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    for (int kb = 0; kb < p.KB; ++kb) {
                        if (!mbar_wait(&sm.full[stage], phase, limit, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_base = smem_addr(smem + SMEM_A + stage * A_STAGE_BYTES);
                        const uint32_t b_base = smem_addr(smem + SMEM_B + stage * B_STAGE_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            umma_bf16_pair(d_tmem, operand_desc<0>(a_base, k),
                                           operand_desc<0>(b_base, k), idesc,
                                           (kb > 0 || k > 0) ? 1u : 0u);
                        umma_commit_pair_mc(&sm.empty[stage], PAIR_MASK);  // stage free in both CTAs
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit_pair_mc(&sm.tfull[acc], PAIR_MASK);  // accumulator ready in both CTAs
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                }
            }
            if (!ok) {
                raise_abort(sm, p.err);
            }
            umma_commit_pair_mc(sm.drain, 0x1);  // every MMA issued so far has completed
            volatile int no_abort = 0;
            mbar_wait(sm.drain, 0, limit, &no_abort);
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int et = threadIdx.x - 64;  // 0..127
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int r = q * 32 + lane;      // accumulator row == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tempty_leader0 = mapa_shared(smem_addr(&sm.tempty[0]), 0);
        const uint32_t tempty_leader1 = mapa_shared(smem_addr(&sm.tempty[1]), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        StoreRing ring;

        for (int u = pair; u < p.units && ok; u += npairs) {
            const Unit t = decode_unit(p, u);
            const int row = t.mt * PM + static_cast<int>(rank) * BM + r;  // row inside this launch
            const bool row_ok = row < p.M;

            long long yv = -1;
            float run_m = -INFINITY, run_s = 0.f, run_t = 0.f, zyv = 0.f;
            bool found = false;
            float lse2 = INFINITY, K1 = 0.f, K2 = 0.f, Bc = 0.f;
            if constexpr (kMode == kFwd) {
                if (row_ok) yv = p.y[row];
            } else {
                if (row_ok) {
                    const int grow = p.row0 + row;
                    yv = p.y[grow];
                    if (yv != p.ignore_index) {
                        const float lse_v = p.lse[grow];
                        const float glp = p.g_lp ? p.g_lp[grow] : 0.f;
                        const float gent = (kEnt && p.g_ent) ? p.g_ent[grow] : 0.f;
                        const float spz = kEnt ? (lse_v - p.ent[grow]) : 0.f;  // sum_j p_j z_j
                        const float A = p.scale * gent;
                        Bc = p.scale * glp;
                        K1 = A * spz - Bc;
                        K2 = -A * p.scale;
                        lse2 = lse_v * LOG2E;
                        if (yv < 0 || yv >= p.V) atomicOr(p.err, ERR_BAD_TARGET);
                    } else {
                        yv = -1;
                    }
                }
            }

            for (int nt = t.n0; nt < t.n1; ++nt) {
                if (!mbar_wait(&sm.tfull[acc], acc_phase, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * BN) + lane_off;
                const int col0 = nt * BN;

                if constexpr (kMode == kFwd) {
                    const int nvalid = min(BN, p.V - col0);
                    const long long tcol = yv - col0;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tbase + c * 32, v);
                        tmem_wait_ld();
                        if (c == BN / 32 - 1) {
                            tc_fence_before();
                            mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
                        }
                        const long long tc = tcol - c * 32;
                        if (tc >= 0 && tc < 32) {
                            zyv = select32(v, static_cast<int>(tc)) * p.scale;
                            found = true;
                        }
                        const int nv = nvalid - c * 32;
                        if (nv <= 0) continue;
                        if (nv >= 32) {
                            // full chunk: packed fp32 pairs halve the FP32 instruction count
                            uint64_t up[16];
                            const uint64_t sc2 = f2_pack(p.scale2, p.scale2);
                            float cmax = -INFINITY;
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                up[j] = f2_mul(f2_pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), sc2);
                                float a, b;
                                f2_unpack(up[j], a, b);
                                cmax = fmax3(cmax, a, b);
                            }
                            if (cmax > run_m) {
                                const float alpha = ex2_approx(run_m - cmax);
                                if constexpr (kEnt)
                                    run_t = (run_s > 0.f) ? alpha * (run_t + run_s * (run_m - cmax)) : 0.f;
                                run_s *= alpha;
                                run_m = cmax;
                            }
                            const uint64_t negm = f2_pack(-run_m, -run_m);
                            uint64_t sacc = f2_pack(0.f, 0.f), tacc = f2_pack(0.f, 0.f);
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const uint64_t d = f2_add(up[j], negm);
                                float d0, d1;
                                f2_unpack(d, d0, d1);
                                const uint64_t e = f2_pack(ex2_approx(d0), ex2_approx(d1));
                                sacc = f2_add(sacc, e);
                                if constexpr (kEnt) tacc = f2_fma(e, d, tacc);
                            }
                            float s0, s1, t0, t1;
                            f2_unpack(sacc, s0, s1);
                            run_s += s0 + s1;
                            if constexpr (kEnt) {
                                f2_unpack(tacc, t0, t1);
                                run_t += t0 + t1;
                            }
                            continue;
                        }
                        // the vocabulary tail: columns >= V are left out of every sum
                        float uu[32];
                        float cmax = -INFINITY;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            uu[j] = (j < nv) ? __uint_as_float(v[j]) * p.scale2 : -INFINITY;
                            cmax = fmaxf(cmax, uu[j]);
                        }
                        if (cmax > run_m) {
                            // rescale the running sums to the new maximum; a row that
                            // has seen nothing yet (run_s == 0) has nothing to rescale
                            const float alpha = ex2_approx(run_m - cmax);
                            if constexpr (kEnt)
                                run_t = (run_s > 0.f) ? alpha * (run_t + run_s * (run_m - cmax)) : 0.f;
                            run_s *= alpha;
                            run_m = cmax;
                        }
                        float s0 = 0.f, t0 = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (j < nv) {
                                const float d0 = uu[j] - run_m;
                                const float e0 = ex2_approx(d0);
                                s0 += e0;
                                if constexpr (kEnt) t0 = fmaf(e0, d0, t0);
                            }
                        }
                        run_s += s0;
                        if constexpr (kEnt) run_t += t0;
                    }
                } else {
                    // dZ: 4 store boxes of 64 bf16 columns each
#pragma unroll 1
                    for (int b = 0; b < BN / 64; ++b) {
                        const uint32_t box = store_box_acquire(ring, smem, et);
                        uint32_t w[32];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t v[32];
                            tmem_ld_32x32b_x32(tbase + b * 64 + h * 32, v);
                            tmem_wait_ld();
                            if (b == BN / 64 - 1 && h == 1) {
                                tc_fence_before();
                                mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
                            }
                            const int cbase = col0 + b * 64 + h * 32;
                            float dz[32];
                            {
                                // packed fp32 pairs: p = 2^(acc s log2e - LSE2), dz = p (K1 + K2 acc)
                                const uint64_t sc2 = f2_pack(p.scale2, p.scale2);
                                const uint64_t nl = f2_pack(-lse2, -lse2);
                                const uint64_t k1 = f2_pack(K1, K1), k2 = f2_pack(K2, K2);
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    const uint64_t a = f2_pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                                    float x0, x1;
                                    f2_unpack(f2_fma(a, sc2, nl), x0, x1);
                                    const uint64_t pp = f2_pack(ex2_approx(x0), ex2_approx(x1));
                                    f2_unpack(f2_mul(pp, f2_fma(a, k2, k1)), dz[2 * j], dz[2 * j + 1]);
                                }
                            }
                            const long long tc = yv - cbase;
                            if (tc >= 0 && tc < 32) {
                                const uint32_t bit = 1u << static_cast<int>(tc);
#pragma unroll
                                for (int j = 0; j < 32; ++j) dz[j] += ((bit >> j) & 1u) ? Bc : 0.f;
                            }
                            const int nv = p.V - cbase;
                            if (nv < 32) {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (j >= nv) dz[j] = 0.f;
                            }
#pragma unroll
                            for (int j = 0; j < 16; ++j) w[h * 16 + j] = pack_bf16x2(dz[2 * j], dz[2 * j + 1]);
                        }
                        stage_row(box, r, w);
                        store_box_release(ring, smem, et, &tmOut, col0 + b * 64,
                                          t.mt * PM + static_cast<int>(rank) * BM, false);
                    }
                }
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) break;

            if constexpr (kMode == kFwd) {
                if (row_ok) {
                    const size_t o = static_cast<size_t>(t.split) * p.M + row;
                    p.part_m[o] = run_m;
                    p.part_s[o] = run_s;
                    if constexpr (kEnt) p.part_t[o] = run_t;
                    if (found) p.zy[row] = zyv;
                }
            }
        }
        if (!ok) {
            raise_abort(sm, p.err);
        }
        if constexpr (kMode == kDz) {
            if (et == 0) bulk_wait_group<0>();
        }
    }

    pair_epilogue(sm, warp, tmem_base);
}

// ----------------------------------------------- fused backward contractions
//
// dX and dW of one wave in a single persistent launch of CTA pairs.  Units
// [0, units_dx) are dX pair tiles (256 wave rows x 256 hidden columns, K =
// padded vocabulary, row tiles fastest); units [units_dx, units_dx + units_dw)
// are dW pair tiles (256 vocabulary rows x 256 hidden columns, K = wave rows,
// hidden tiles fastest).  The leader CTA's producer takes tickets from a global
// counter, so the long dX tiles start first and the short dW tiles fill the
// tail evenly, and publishes each unit to both CTAs through a shared-memory
// ring (mirrored into the peer with st.shared::cluster) guarded by mbarriers:
// sched_full in each CTA, sched_empty in the leader (counting the leader's MMA
// thread, the peer's producer and both CTAs' epilogue threads).

struct BwdParams {
    int units_dx, units_dw;
    int Mt_dx;   // 256-row pair tiles of the wave
    int GM_dx;   // dX tiles are ordered in groups of GM_dx row tiles (L2 reuse of dZ rows and W columns)
    int Nt;      // 256-column tiles of H
    int KB_dx;   // K blocks of the padded vocabulary
    int KB_dw;   // K blocks of the wave rows
    int dw_add;  // 0: store dW tiles, 1: add them to dW
    unsigned long long* ticket;  // global counter (zeroed by the call)
    unsigned long long ticket_base;
    int* err;
    unsigned long long wait_limit_ns;
};

struct BwdUnit {
    int dw, mt, nt, kb_count;
};

__device__ __forceinline__ BwdUnit decode_bwd(const BwdParams& p, int u) {
    BwdUnit t;
    if (u < p.units_dx) {
        t.dw = 0;
        const int per_group = p.GM_dx * p.Nt;
        const int g = u / per_group;
        const int gm = min(p.GM_dx, p.Mt_dx - g * p.GM_dx);
        const int r = u - g * per_group;
        t.nt = r / gm;
        t.mt = g * p.GM_dx + (r - t.nt * gm);
        t.kb_count = p.KB_dx;
    } else {
        const int v = u - p.units_dx;
        t.dw = 1;
        t.mt = v / p.Nt;
        t.nt = v - t.mt * p.Nt;
        t.kb_count = p.KB_dw;
    }
    return t;
}

// kDxF32: dX boxes in fp32 (else bf16).  kDwBf16: dW boxes in bf16, stored
// (single wave, no accumulation; else fp32, stored or added).
template <bool kDxF32, bool kDwBf16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    flp_bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmDzK,   // dZ, K-major A (dX)
                        const __grid_constant__ CUtensorMap tmWmn,   // W, MN-major B (dX)
                        const __grid_constant__ CUtensorMap tmDzMn,  // dZ, MN-major A (dW)
                        const __grid_constant__ CUtensorMap tmXmn,   // X[wave], MN-major B (dW)
                        const __grid_constant__ CUtensorMap tmDx,    // dX[wave] store boxes
                        const __grid_constant__ CUtensorMap tmDw,    // dW store / add boxes
                        const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = smem_layout(smem_raw);
    uint8_t* smem = sm.base;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int total = p.units_dx + p.units_dw;
    const int rofs = static_cast<int>(rank) * BM;  // this CTA's rows / columns inside a pair tile

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmDzK);
        tma_prefetch_desc(&tmWmn);
        tma_prefetch_desc(&tmDzMn);
        tma_prefetch_desc(&tmXmn);
        tma_prefetch_desc(&tmDx);
        tma_prefetch_desc(&tmDw);
    }
    const uint32_t tmem_base = pair_prologue(sm, warp);
    const uint64_t limit = p.wait_limit_ns;
    volatile int* abort_flag = sm.abort_flag;

    if (warp == 0) {
        // ------------------------------------------- scheduler + TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // the leader holds the next ticket one unit ahead, so the global
            // atomic's latency overlaps the current unit's loads
            unsigned long long next_tk = leader ? atomicAdd(p.ticket, 1ull) : 0ull;
            // The leader keeps one unit published ahead of the one it loads, so
            // the peer finds the next unit in its ring when it needs it.
            int published = 0;
            bool ended = false;  // the terminating (-1) unit is in the ring
            for (int it = 0; ok; ++it) {
                const int slot = it % SCHED_SLOTS;
                const uint32_t sph = static_cast<uint32_t>(it / SCHED_SLOTS) & 1u;
                int u;
                if (leader) {
                    while (!ended && published < it + 2) {
                        const int ps = published % SCHED_SLOTS;
                        const uint32_t pph = static_cast<uint32_t>(published / SCHED_SLOTS) & 1u;
                        if (!mbar_wait(&sm.sched_empty[ps], pph ^ 1u, limit, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const unsigned long long tk = next_tk - p.ticket_base;
                        const int pu = (tk < static_cast<unsigned long long>(total)) ? static_cast<int>(tk) : -1;
                        if (pu >= 0) next_tk = atomicAdd(p.ticket, 1ull);
                        sm.sched_val[ps] = pu;
                        st_shared_cluster_u32(mapa_shared(smem_addr(const_cast<int*>(&sm.sched_val[ps])), 1),
                                              static_cast<uint32_t>(pu));
                        mbar_arrive(&sm.sched_full[ps]);
                        mbar_arrive_cluster(mapa_shared(smem_addr(&sm.sched_full[ps]), 1));
                        ++published;
                        if (pu < 0) ended = true;
                    }
                    if (!ok) break;
                    u = sm.sched_val[slot];  // written by this thread; not reused before `published` passes it + 4
                } else {
                    if (!mbar_wait<true>(&sm.sched_full[slot], sph, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    u = sm.sched_val[slot];
                    mbar_arrive_cluster(mapa_shared(smem_addr(&sm.sched_empty[slot]), 0));
                }
                if (u < 0) break;
                const BwdUnit t = decode_bwd(p, u);
                for (int kb = 0; kb < t.kb_count; ++kb) {
                    if (!mbar_wait(&sm.empty[stage], phase ^ 1u, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(&sm.full[stage], PAIR_STAGE_TX);
                    const uint32_t bar = mapa_shared(smem_addr(&sm.full[stage]), 0);
                    uint8_t* a_dst = smem + SMEM_A + stage * A_STAGE_BYTES;
                    uint8_t* b_dst = smem + SMEM_B + stage * B_STAGE_BYTES;
                    if (!t.dw) {
                        tma_load_2d_pair(a_dst, &tmDzK, kb * BK, t.mt * PM + rofs, bar);
#pragma unroll
                        for (int j = 0; j < BNH / 64; ++j)
                            tma_load_2d_pair(b_dst + j * 8192, &tmWmn, t.nt * BN + rofs + j * 64, kb * BK, bar);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d_pair(a_dst + j * 8192, &tmDzMn, t.mt * PM + rofs + j * 64, kb * BK, bar);
#pragma unroll
                        for (int j = 0; j < BNH / 64; ++j)
                            tma_load_2d_pair(b_dst + j * 8192, &tmXmn, t.nt * BN + rofs + j * 64, kb * BK, bar);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                raise_abort(sm, p.err);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------- MMA issuer (leader)
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            constexpr uint32_t idesc_dx = idesc_bf16_f32(PM, BN, 0, 1);
            constexpr uint32_t idesc_dw = idesc_bf16_f32(PM, BN, 1, 1);
            for (int it = 0; ok; ++it) {
                const int slot = it % SCHED_SLOTS;
                const uint32_t sph = static_cast<uint32_t>(it / SCHED_SLOTS) & 1u;
                if (!mbar_wait(&sm.sched_full[slot], sph, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                const int u = sm.sched_val[slot];
                mbar_arrive(&sm.sched_empty[slot]);
                if (u < 0) break;
                const BwdUnit t = decode_bwd(p, u);
                if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < t.kb_count; ++kb) {
                    if (!mbar_wait(&sm.full[stage], phase, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_addr(smem + SMEM_A + stage * A_STAGE_BYTES);
                    const uint32_t b_base = smem_addr(smem + SMEM_B + stage * B_STAGE_BYTES);
                    if (!t.dw) {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            umma_bf16_pair(d_tmem, operand_desc<0>(a_base, k), operand_desc<1>(b_base, k),
                                           idesc_dx, (kb > 0 || k > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            umma_bf16_pair(d_tmem, operand_desc<1>(a_base, k), operand_desc<1>(b_base, k),
                                           idesc_dw, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit_pair_mc(&sm.empty[stage], PAIR_MASK);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(&sm.tfull[acc], PAIR_MASK);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                raise_abort(sm, p.err);
            }
            umma_commit_pair_mc(sm.drain, 0x1);
            volatile int no_abort = 0;
            mbar_wait(sm.drain, 0, limit, &no_abort);
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int et = threadIdx.x - 64;
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tempty_leader0 = mapa_shared(smem_addr(&sm.tempty[0]), 0);
        const uint32_t tempty_leader1 = mapa_shared(smem_addr(&sm.tempty[1]), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        StoreRing ring;
        for (int it = 0; ok; ++it) {
            const int slot = it % SCHED_SLOTS;
            const uint32_t sph = static_cast<uint32_t>(it / SCHED_SLOTS) & 1u;
            if (!mbar_wait<true>(&sm.sched_full[slot], sph, limit, abort_flag)) {
                ok = false;
                break;
            }
            const int u = sm.sched_val[slot];
            mbar_arrive_cluster(mapa_shared(smem_addr(&sm.sched_empty[slot]), 0));
            if (u < 0) break;
            const BwdUnit t = decode_bwd(p, u);
            if (!mbar_wait(&sm.tfull[acc], acc_phase, limit, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * BN) + lane_off;
            const int col0 = t.nt * BN;
            const int row0 = t.mt * PM + rofs;
            const bool bf16_out = t.dw ? kDwBf16 : !kDxF32;
            if (bf16_out) {
                const CUtensorMap* out = t.dw ? &tmDw : &tmDx;
#pragma unroll 1
                for (int b = 0; b < BN / 64; ++b) {
                    const uint32_t box = store_box_acquire(ring, smem, et);
                    uint32_t w[32];
                    tmem_row64_to_bf16(tbase + b * 64, w);
                    if (b == BN / 64 - 1) {
                        tc_fence_before();
                        mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
                    }
                    stage_row(box, r, w);
                    store_box_release(ring, smem, et, out, col0 + b * 64, row0, false);
                }
            } else {
                const CUtensorMap* out = t.dw ? &tmDw : &tmDx;
                const bool add = t.dw && p.dw_add;
#pragma unroll 1
                for (int b = 0; b < BN / 32; ++b) {
                    const uint32_t box = store_box_acquire(ring, smem, et);
                    uint32_t w[32];
                    tmem_ld_32x32b_x32(tbase + b * 32, w);
                    tmem_wait_ld();
                    if (b == BN / 32 - 1) {
                        tc_fence_before();
                        mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
                    }
                    stage_row(box, r, w);
                    store_box_release(ring, smem, et, out, col0 + b * 32, row0, add);
                }
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok) {
            raise_abort(sm, p.err);
        }
        if (et == 0) bulk_wait_group<0>();
    }

    pair_epilogue(sm, warp, tmem_base);
}

// ------------------------------------------------------------- split merge

struct MergeParams {
    int M, S, V;
    long long ignore_index;
    int compute_entropy;
    const long long* y;
    const float* part_m;
    const float* part_s;
    const float* part_t;
    const float* zy;
    float* logprob;
    float* lse;
    float* entropy;
    int* err;
};

// Online combination of two (max, sum-exp, entropy sum) triples in base-2
// units: the sums are rescaled to the larger max; a triple with sum 0 (a split
// that saw no column) contributes nothing, so no 0 * inf arises.
struct Stats {
    float m, s, t;
};

__device__ __forceinline__ Stats combine(Stats a, Stats b) {
    if (!(b.s > 0.f)) return a;
    if (!(a.s > 0.f)) return b;
    const float m = fmaxf(a.m, b.m);
    const float da = a.m - m, db = b.m - m;
    const float ea = exp2f(da), eb = exp2f(db);
    Stats r;
    r.m = m;
    r.s = a.s * ea + b.s * eb;
    r.t = (a.t + a.s * da) * ea + (b.t + b.s * db) * eb;
    return r;
}

constexpr int MERGE_ROWS = 32;   // rows per block (one per lane)
constexpr int MERGE_WAYS = 8;    // warps per block; warp w reads splits w, w + 8, ...

// Combines the per-split partials of each row into the final lse / logprob /
// entropy (the "reduced" and "result" stages kept in buffers separate from the
// raw partials).  Each warp reads a stripe of splits for 32 consecutive rows
// (coalesced), the stripes are combined through shared memory.  Base-2 units
// inside, natural log out.
__global__ void __launch_bounds__(MERGE_ROWS * MERGE_WAYS) flp_merge_kernel(const MergeParams p) {
    __shared__ Stats part[MERGE_WAYS][MERGE_ROWS];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int i = blockIdx.x * MERGE_ROWS + lane;
    Stats acc{-INFINITY, 0.f, 0.f};
    if (i < p.M) {
        for (int k = w; k < p.S; k += MERGE_WAYS) {
            const size_t o = static_cast<size_t>(k) * p.M + i;
            Stats v{p.part_m[o], p.part_s[o], p.compute_entropy ? p.part_t[o] : 0.f};
            acc = combine(acc, v);
        }
    }
    part[w][lane] = acc;
    __syncthreads();
    if (w != 0 || i >= p.M) return;
#pragma unroll
    for (int j = 1; j < MERGE_WAYS; ++j) acc = combine(acc, part[j][lane]);
    const float l2s = log2f(acc.s);
    const float lse = (acc.m + l2s) * LN2;
    p.lse[i] = lse;
    const long long yv = p.y[i];
    float lp, ent = p.compute_entropy ? (l2s - acc.t / acc.s) * LN2 : 0.f;
    if (yv == p.ignore_index) {
        lp = 0.f;
        ent = 0.f;
    } else if (yv < 0 || yv >= p.V) {
        lp = __int_as_float(0x7fc00000);
        atomicOr(p.err, ERR_BAD_TARGET);
    } else {
        lp = p.zy[i] - lse;
    }
    p.logprob[i] = lp;
    if (p.compute_entropy) p.entropy[i] = ent;
}

}  // namespace flp
