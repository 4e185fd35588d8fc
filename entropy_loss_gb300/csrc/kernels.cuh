// kernels.cuh - sm_103a kernels of the fused linear log-prob / cross-entropy head.
//
// Every contraction of the path runs on CTA pairs (clusters of two CTAs on two
// SMs) that share an output tile: tcgen05.mma.cta_group::2 with M = 256 (128
// rows of A in each CTA) and N = 256 (B split along N, 128 rows in each CTA),
// fp32 accumulators in both CTAs' TMEM.  For a 256 x 256 tile each SM loads
// 16 KiB of A and 16 KiB of B per 64-deep K step for 2 * 128 * 256 * 64 MACs;
// a wide 256 x 512 tile (both accumulators) loads 48 KiB for twice that.
//
//   flp_fwd_kernel   : z = s X W^T tiles -> online max / sum-exp / (entropy) /
//                      target pick per row -> raw per-split partials
//   flp_merge_kernel : per-split partials -> lse, logprob, entropy
//   flp_dz_kernel    : (bwd.cuh) the dZ tiles of the split backward schedules
//   flp_bwd_kernel   : (bwd.cuh) dX and dW tiles, and all tiles of the fused one
//
// This file holds the pieces every pair kernel shares (shared-memory layout,
// barrier set-up and teardown, descriptors, store boxes, the wide tiles'
// producer step and staggered MMA issue), the forward and the merge.
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
// The forward, the dZ kernel and the backward's dX + dW launch run wide tiles
// instead: 256 rows x 512 columns, one per pair, both accumulators (half h of
// the columns in accumulator h), so each SM loads 16 KiB of A and 32 KiB of B
// per K step for twice the MACs (25 % fewer operand bytes per MAC).  They have
// two epilogue groups of four warps (warps 2..5 drain half 0, warps 6..9 half
// 1; 320 threads), and the MMA issuer staggers the halves at both ends of a
// tile so that one half's epilogue runs under the other half's MMAs.
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
constexpr int WIDE_THREADS = 64 + 2 * EPI_THREADS;  // wide-tile kernels (forward, dZ, dX + dW): two epilogue groups of four warps
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

// Shared-memory slots.  Normal tiles: STAGES slots of 16 KiB of A and 16 KiB
// of B (A slots first, then B slots).  Wide tiles (the forward's, and dX tiles
// of the backward): STAGES_W slots of 48 KiB (A, then the B halves of the two
// 256-column sub-tiles), over the same bytes.
constexpr int STAGES_W = 4;
constexpr uint32_t STAGE_W_BYTES = A_STAGE_BYTES + 2 * B_STAGE_BYTES;
constexpr uint32_t PAIR_STAGE_TX_W = 2 * STAGE_W_BYTES;
static_assert(STAGES_W * STAGE_W_BYTES <= SMEM_STG, "wide slots must fit the pipeline region");

__device__ __forceinline__ uint32_t slot_a(bool wide, int s) {
    return wide ? s * STAGE_W_BYTES : SMEM_A + s * A_STAGE_BYTES;
}
__device__ __forceinline__ uint32_t slot_b(bool wide, int s) {
    return wide ? s * STAGE_W_BYTES + A_STAGE_BYTES : SMEM_B + s * B_STAGE_BYTES;
}

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
// sched_arrivals: arrivals that free a slot of the unit hand-off ring (the
// peer's producer, the MMA issuer and every epilogue thread of both CTAs).
__device__ __forceinline__ uint32_t pair_prologue(const Smem& sm, int warp,
                                                  uint32_t sched_arrivals = 2 + 2 * EPI_THREADS) {
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
            mbar_init(&sm.sched_empty[s], sched_arrivals);
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

// Narrow store boxes: 128 rows x 64 bytes (32 bf16 or 16 fp32 columns,
// 64-byte swizzle), two per epilogue group, so that two groups fit the store
// region.  One box of this thread's row (16 words) is staged and stored (or
// added) in its group's ring, with one named barrier per box: before it,
// thread 0 of the group waits until every earlier bulk store has finished
// reading, so after it the other box (read by the previous store) may be
// rewritten by the next call while this box's store runs.
constexpr uint32_t NBOX_BYTES = BM * 64;
static_assert(2 * 2 * NBOX_BYTES <= NUM_STG * STG_BYTES, "two narrow boxes per epilogue group");

__device__ __forceinline__ void narrow_box_store(StoreRing& ring, uint8_t* box0, uint32_t bar_id, int et, int r,
                                                 const uint32_t* w, const CUtensorMap* out, int x, int y,
                                                 bool add) {
    const uint32_t buf = ring.n & 1u;
    // box buf was last read by the store two boxes back, which thread 0
    // waited for before the previous call's barrier
    uint8_t* box = box0 + buf * NBOX_BYTES;
    const uint32_t row_addr = smem_addr(box) + r * 64;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        st_shared_v4(row_addr + ((c ^ ((r >> 1) & 3)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    fence_proxy_async_smem();
    if (et == 0) bulk_wait_group_read<0>();  // the other box is free again after the barrier
    named_bar_sync(bar_id, EPI_THREADS);
    if (et == 0) {
        if (add)
            tma_reduce_add_2d(out, box, x, y);
        else
            tma_store_2d(out, box, x, y);
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

// ------------------------------------------------------ wide (256 x 512) tiles

// k-blocks issued half by half at each end of a wide tile (at most the number
// of wide slots: those k-blocks' stages stay held until both halves ran)
constexpr int WIDE_EDGE = STAGES_W;

// Producer: one 64-deep k-block of a wide tile whose operands are both K-major
// into wide slot `stage`: this CTA's 128 rows of A (from row a_row) and its
// 128-row halves of the two 256-row B sub-tiles (from rows b_row, b_row + 256).
__device__ __forceinline__ void load_wide_kblock(const Smem& sm, int stage, bool leader,
                                                 const CUtensorMap* tmA, int a_row,
                                                 const CUtensorMap* tmB, int b_row, int kb) {
    if (leader) mbar_arrive_expect_tx(&sm.full[stage], PAIR_STAGE_TX_W);
    const uint32_t bar = mapa_shared(smem_addr(&sm.full[stage]), 0);
    tma_load_2d_pair(sm.base + slot_a(true, stage), tmA, kb * BK, a_row, bar);
#pragma unroll
    for (int h = 0; h < 2; ++h)
        tma_load_2d_pair(sm.base + slot_b(true, stage) + h * B_STAGE_BYTES, tmB, kb * BK, b_row + h * BN, bar);
}

// MMA issuer: every MMA of one wide tile with K-major operands (KB k-blocks),
// half h into accumulator h, then tfull[h] per half.  `gk` counts the
// k-blocks consumed so far (slot gk % STAGES_W, fill parity
// (gk / STAGES_W) & 1) and advances by KB; acc_phase is this tile's use
// parity of the accumulators.  The first and last WIDE_EDGE k-blocks are
// issued half by half: at the end of the tile half 0 completes (and its
// epilogue starts) while the half-1 MMAs of those k-blocks still run, and at
// the start half 0 fills while the previous tile's half 1 is still drained.
// Returns false when a wait ran out.
__device__ __forceinline__ bool wide_tile_mma(const Smem& sm, uint32_t tmem_base, uint32_t& gk,
                                              uint32_t acc_phase, int KB, uint64_t limit,
                                              volatile int* abort_flag) {
    constexpr uint32_t idesc = idesc_bf16_f32(PM, BN, 0, 0);
    auto issue = [&](uint32_t g, int h, int kb) {
        const int s = static_cast<int>(g % STAGES_W);
        const uint32_t a_base = smem_addr(sm.base + slot_a(true, s));
        const uint32_t b_base = smem_addr(sm.base + slot_b(true, s)) + h * B_STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k)
            umma_bf16_pair(tmem_base + static_cast<uint32_t>(h * BN), operand_desc<0>(a_base, k),
                           operand_desc<0>(b_base, k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
    };
    auto wait_full = [&](uint32_t g) {
        if (!mbar_wait(&sm.full[g % STAGES_W], (g / STAGES_W) & 1u, limit, abort_flag)) return false;
        tc_fence_after();
        return true;
    };
    auto release = [&](uint32_t g) {
        umma_commit_pair_mc(&sm.empty[g % STAGES_W], PAIR_MASK);  // stage free in both CTAs
    };
    const int head = min(WIDE_EDGE, KB);
    const int tail0 = max(head, KB - WIDE_EDGE);
    if (!mbar_wait(&sm.tempty[0], acc_phase ^ 1u, limit, abort_flag)) return false;
    tc_fence_after();
    for (int kb = 0; kb < head; ++kb) {
        if (!wait_full(gk + kb)) return false;
        issue(gk + kb, 0, kb);
    }
    if (head == KB) umma_commit_pair_mc(&sm.tfull[0], PAIR_MASK);
    if (!mbar_wait(&sm.tempty[1], acc_phase ^ 1u, limit, abort_flag)) return false;
    tc_fence_after();
    for (int kb = 0; kb < head; ++kb) {
        issue(gk + kb, 1, kb);
        release(gk + kb);
    }
    for (int kb = head; kb < tail0; ++kb) {
        if (!wait_full(gk + kb)) return false;
        issue(gk + kb, 0, kb);
        issue(gk + kb, 1, kb);
        release(gk + kb);
    }
    for (int kb = tail0; kb < KB; ++kb) {
        if (!wait_full(gk + kb)) return false;
        issue(gk + kb, 0, kb);
    }
    if (head < KB) umma_commit_pair_mc(&sm.tfull[0], PAIR_MASK);  // half 0 ready in both CTAs
    for (int kb = tail0; kb < KB; ++kb) {
        issue(gk + kb, 1, kb);
        release(gk + kb);
    }
    umma_commit_pair_mc(&sm.tfull[1], PAIR_MASK);  // half 1 ready in both CTAs
    gk += static_cast<uint32_t>(KB);
    return true;
}

// ------------------------------------------------------------ forward kernel

struct FwdParams {
    // schedule: units are runs [n0, n1) of 512-column tiles sharing one 256-row pair tile;
    // each unit writes two partials per row (one per 256-column half): S * 2 in all
    int units, Mt, Nt, S, tps, GM;
    int KB;    // K blocks of 64 (H / 64, rounded up)
    int M;     // rows
    int V;     // vocabulary size (column mask)
    long long ignore_index;
    float scale;   // s
    float scale2;  // s * log2(e)
    const long long* y;
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
__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int u) {
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

template <bool kEnt>
__global__ void __launch_bounds__(WIDE_THREADS, 1)
    flp_fwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = smem_layout(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (threadIdx.x == 0) griddep_launch_dependents();  // the next launch may be scheduled early
    const uint32_t tmem_base = pair_prologue(sm, warp);
    griddep_wait();  // the previous launch's results (dZ, the error word) are complete from here on
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
                        load_wide_kblock(sm, stage, leader, &tmA, t.mt * PM + static_cast<int>(rank) * BM,
                                         &tmB, nt * 2 * BN + static_cast<int>(rank) * BNH, kb);
                        ++issued;
                        if (++stage == STAGES_W) {
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
            uint32_t gk = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = pair; u < p.units && ok; u += npairs) {
                const Unit t = decode_unit(p, u);
                for (int nt = t.n0; nt < t.n1 && ok; ++nt) {
                    ok = wide_tile_mma(sm, tmem_base, gk, acc_phase, p.KB, limit, abort_flag);
                    acc_phase ^= 1u;
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
        // two groups of four warps: group g drains accumulator g, the
        // 256-column half g of every 512-column tile
        const int g = (warp - 2) >> 2;
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int r = q * 32 + lane;      // accumulator row == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tempty_leader = mapa_shared(smem_addr(&sm.tempty[g]), 0);
        const int acc = g;
        uint32_t acc_phase = 0;
        bool ok = true;

        for (int u = pair; u < p.units && ok; u += npairs) {
            const Unit t = decode_unit(p, u);
            const int row = t.mt * PM + static_cast<int>(rank) * BM + r;
            const bool row_ok = row < p.M;
            const long long yv = row_ok ? p.y[row] : -1;
            float run_m = -INFINITY, run_s = 0.f, run_t = 0.f, zyv = 0.f;
            bool found = false;

            for (int nt = t.n0; nt < t.n1; ++nt) {
                if (!mbar_wait(&sm.tfull[acc], acc_phase, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * BN) + lane_off;
                const int col0 = nt * 2 * BN + g * BN;
                const int nvalid = min(BN, p.V - col0);
                const long long tcol = yv - col0;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_wait_ld();
                    if (c == BN / 32 - 1) {
                        tc_fence_before();
                        mbar_arrive_cluster(tempty_leader);
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
                acc_phase ^= 1u;
            }
            if (!ok) break;

            if (row_ok) {
                const size_t o = static_cast<size_t>(2 * t.split + g) * p.M + row;
                p.part_m[o] = run_m;
                p.part_s[o] = run_s;
                if constexpr (kEnt) p.part_t[o] = run_t;
                if (found) p.zy[row] = zyv;
            }
        }
        if (!ok) {
            raise_abort(sm, p.err);
        }
    }

    pair_epilogue(sm, warp, tmem_base);
}

// ---------------------------------------------------------- fp32 -> bf16

// dst[i] = bf16(src[i]) (round to nearest even): the vocabulary-split
// backward's fp32 dX, accumulated over the chunks, rounded once.  n may be
// any size; the 16-byte vector path runs while 8 elements remain.
__global__ void __launch_bounds__(256) flp_round_bf16_kernel(const float* __restrict__ src,
                                                             uint16_t* __restrict__ dst, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 8;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; i < n; i += stride) {
        if (i + 8 <= n) {
            const float4 a = *reinterpret_cast<const float4*>(src + i);
            const float4 b = *reinterpret_cast<const float4*>(src + i + 4);
            uint4 o;
            o.x = pack_bf16x2(a.x, a.y);
            o.y = pack_bf16x2(a.z, a.w);
            o.z = pack_bf16x2(b.x, b.y);
            o.w = pack_bf16x2(b.z, b.w);
            *reinterpret_cast<uint4*>(dst + i) = o;
        } else {
            for (int64_t j = i; j < n; ++j) dst[j] = static_cast<uint16_t>(pack_bf16x2(src[j], 0.f) & 0xFFFFu);
        }
    }
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
constexpr int MERGE_BATCH = 8;   // splits whose loads a warp has in flight at once

// Combines the per-split partials of each row into the final lse / logprob /
// entropy (the "reduced" and "result" stages kept in buffers separate from the
// raw partials).  Each warp reads a stripe of splits for 32 consecutive rows
// (coalesced), the stripes are combined through shared memory.  Base-2 units
// inside, natural log out.  When the forward tile kernel gave up on a wait
// (timeout bit in the error word) its partials are incomplete: every output
// row is then NaN, so that no stale or partial value passes for a result.
__global__ void __launch_bounds__(MERGE_ROWS * MERGE_WAYS) flp_merge_kernel(const MergeParams p) {
    __shared__ Stats part[MERGE_WAYS][MERGE_ROWS];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int i = blockIdx.x * MERGE_ROWS + lane;
    griddep_wait();  // the forward tile kernel's partials and error word are complete
    if (*reinterpret_cast<volatile const int*>(p.err) & ERR_TIMEOUT) {
        if (w == 0 && i < p.M) {
            const float nan = __int_as_float(0x7fc00000);
            p.lse[i] = nan;
            p.logprob[i] = nan;
            if (p.compute_entropy) p.entropy[i] = nan;
        }
        return;
    }
    Stats acc{-INFINITY, 0.f, 0.f};
    if (i < p.M) {
        // splits w, w + 8, w + 16, ... in order; the loads of MERGE_BATCH of
        // them are issued before any is combined (the loop is latency-bound)
        for (int k0 = w; k0 < p.S; k0 += MERGE_BATCH * MERGE_WAYS) {
            Stats v[MERGE_BATCH];
#pragma unroll
            for (int j = 0; j < MERGE_BATCH; ++j) {
                const int k = k0 + j * MERGE_WAYS;
                v[j] = Stats{-INFINITY, 0.f, 0.f};
                if (k < p.S) {
                    const size_t o = static_cast<size_t>(k) * p.M + i;
                    v[j] = Stats{p.part_m[o], p.part_s[o], p.compute_entropy ? p.part_t[o] : 0.f};
                }
            }
#pragma unroll
            for (int j = 0; j < MERGE_BATCH; ++j) acc = combine(acc, v[j]);
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
