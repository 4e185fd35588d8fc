// bwd.cuh - the backward of the fused linear log-prob head on CTA pairs.
//
// Two persistent kernels.  flp_bwd_kernel (instantiated per set of tile kinds
// a launch holds) runs pair tiles of three kinds, 256 x 256 unless noted:
//   dZ : the logits tile recomputed (K = H), then
//        dZ = s [g_lp (onehot - p) + g_ent p (sum_j p_j z_j - z)]  in bf16,
//        TMA-stored to the wave's dZ buffer (rows of the wave x padded V)
//   dX : dX[wave] tile = dZ W        (K = padded vocabulary; W read MN-major)
//   dW : dW tile (+)= dZ^T X[wave]   (K = wave rows; both operands MN-major)
// dX tiles, and the split schedules' dW tiles, are 256 x 512 when H allows:
// two N = 256 MMAs share each A stage, so an SM loads 48 KiB per 64-deep K
// step for twice the MACs (the mainloops are bound by how fast an SM ingests
// operands from L2), with the two halves staggered at the tile ends.
// flp_dz_kernel runs the split schedules' dZ launch on 256 x 512 tiles, the
// forward's mainloop with a dZ epilogue.
// The leader CTA of each pair takes tickets from a global counter and maps
// them to units through a schedule of segments that the host lays down, then
// publishes each unit to both CTAs' roles through a shared-memory ring.  A
// launch of equal-length units (the dZ launch) instead runs a static
// round-robin that every role computes for itself.
//
// Three schedules drive them (the host picks one per call):
//   split : per row wave, one flp_dz_kernel launch with the wave's dZ tiles,
//           then one flp_bwd_kernel launch with its dX tiles (long, first)
//           and dW tiles (short, filling the tail); the kernel boundary
//           orders the phases.
//   vsplit: all rows in one wave and the vocabulary in chunks: per chunk the
//           same two launches over the chunk's columns; dX accumulates over
//           the chunks in fp32, each dW tile is written once (K = all rows).
//   fused : every wave in one flp_bwd_kernel launch (256 x 256 dZ and dW
//           tiles).  A dX tile waits until the dZ tiles of its rows are
//           stored, a dW tile until those of its vocabulary column are; from
//           the second wave on, a dZ tile waits until the previous wave's dX
//           and dW tiles that read its buffer slot are done, and a dW tile
//           until the previous wave's add into the same dW rows is.  The
//           counters live in the workspace; every wait is on a ticket handed
//           out earlier, so the lowest unfinished ticket can always proceed,
//           and every wait is bounded in time.
// Every schedule computes each 256 x 256 block of an output with the same
// instructions in the same K order (a wide tile's halves are two such
// blocks), so their results agree bit for bit.
#pragma once
#include "kernels.cuh"

namespace flp {

enum UnitKind : int { kUnitDz = 0, kUnitDx = 1, kUnitDw = 2 };

// A segment is a run of consecutive tickets that decode to one pattern:
//   kSegDz   : dZ tiles of row tiles [a0, a0 + an), vocabulary tiles from b0
//              on; vocabulary outer, rows inner (the rows share each W tile)
//   kSegDx   : dX tiles of row tiles [a0, a0 + an); hidden tiles outer
//   kSegDw   : dW tiles of vocabulary tiles from b0 on; hidden tiles inner
//   kSegDzDw : blocks of (the an dZ tiles of vocabulary tile b0 + c, then the
//              Nh dW tiles of vocabulary tile b0 + c - lag), so that a dW
//              tile reads a dZ column written a few blocks earlier (in L2)
//   kSegDx2  : wide (256 x 512) dX tiles of row tiles [a0, a0 + an); 512-column
//              hidden tiles outer
//   kSegDz2  : wide (256 x 512) dZ tiles of row tiles [a0, a0 + an), vocabulary
//              tiles (b0 + 2c, b0 + 2c + 1) for c = 0, 1, ...; vocabulary outer
//              (run by flp_dz_kernel, never mixed with other kinds)
//   kSegDw2  : wide (256 x 512) dW tiles of vocabulary tiles from b0 on;
//              512-column hidden tiles inner
enum SegKind : int { kSegDz = 0, kSegDx = 1, kSegDw = 2, kSegDzDw = 3, kSegDx2 = 4, kSegDz2 = 5, kSegDw2 = 6 };

struct BwdSeg {
    int start;  // first ticket
    int kind;
    int wave;
    int a0, an;
    int b0;
    int lag;
};

constexpr int MAX_SEGS = 160;

struct BwdParams {
    int total;       // tickets of this launch
    int nseg;
    int M;           // rows covered by the row tensor maps of this launch
    int V;           // vocabulary size (column mask)
    int chunk;       // rows of a full wave; wave w starts at row w * chunk
    int nwaves;
    int Mt_full;     // 256-row pair tiles of a full wave
    int Vt;          // 256-column tiles of the padded vocabulary
    int Nh;          // 256-column tiles of H
    int Ndx;         // dX tiles per row tile (Nh, or Nh / 2 wide tiles)
    int KB_h;        // 64-deep K blocks of H (dZ tiles)
    int KB_v;        // 64-deep K blocks of the padded vocabulary chunk (dX tiles)
    int deps;        // 1: the fused schedule's dependency counters are live
    int static_order;  // 1: pair p runs units p, p + pairs, ... (no tickets, no hand-off ring)
    int dw_add0;     // wave 0 adds into dW (accumulate); later waves always add
    int vt0;         // first vocabulary tile of this launch's vocabulary chunk (0: all of V)
    int vt_end;      // end of this launch's vocabulary tiles (wide dZ tiles store no half at or past it)
    int dx_add;      // dX tiles add into their (fp32) output (later vocabulary chunks)
    int dx_f32;      // dX boxes in fp32 (else bf16)
    int dw_bf16;     // dW boxes in bf16 (one wave, no accumulation; else fp32)
    int ent;         // the entropy term is part of the upstream gradient
    long long ignore_index;
    float scale;     // s
    float scale2;    // s * log2(e)
    const long long* y;
    const float* lse;
    const float* ent_v;
    const float* g_lp;
    const float* g_ent;
    uint32_t* row_dz;   // [Mt_full] dZ tile stores finished per row tile (2 per tile: one per CTA)
    uint32_t* col_dz;   // [Vt]      ... per vocabulary tile
    uint32_t* dx_done;  // [Mt_full] dX tiles finished per row tile (2 per tile: one per CTA)
    uint32_t* dw_done;  // [Vt]      dW tiles finished per vocabulary tile (2 per tile)
    unsigned long long* ticket;
    unsigned long long ticket_base;
    int* err;
    unsigned long long wait_limit_ns;
    int debug_stop_at;  // flp_dz_kernel self-test: 0 off; n > 0: its producers stop after n - 1 stages
    BwdSeg seg[MAX_SEGS];
};

struct BUnit {
    int kind, wave;
    int mt;    // dZ, dX: row tile of the wave; dW: vocabulary tile
    int nt;    // dZ: vocabulary tile (the first of two for a wide one); dX, dW: hidden tile
               // (of 512 columns for a wide one)
    int wide;  // a 256 x 512 tile
};

__host__ __device__ __forceinline__ BUnit decode_bwd(const BwdParams& p, int u) {
    int lo = 0, hi = p.nseg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].start <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    const BwdSeg& s = p.seg[lo];
    const int off = u - s.start;
    BUnit t;
    t.wave = s.wave;
    t.wide = 0;
    if (s.kind == kSegDz) {
        t.kind = kUnitDz;
        t.nt = s.b0 + off / s.an;
        t.mt = s.a0 + off % s.an;
    } else if (s.kind == kSegDx) {
        t.kind = kUnitDx;
        t.nt = off / s.an;
        t.mt = s.a0 + off % s.an;
    } else if (s.kind == kSegDw) {
        t.kind = kUnitDw;
        t.mt = s.b0 + off / p.Nh;
        t.nt = off % p.Nh;
    } else if (s.kind == kSegDx2) {
        t.kind = kUnitDx;
        t.wide = 1;
        t.nt = off / s.an;
        t.mt = s.a0 + off % s.an;
    } else if (s.kind == kSegDz2) {
        t.kind = kUnitDz;
        t.wide = 1;
        t.nt = s.b0 + 2 * (off / s.an);
        t.mt = s.a0 + off % s.an;
    } else if (s.kind == kSegDw2) {
        t.kind = kUnitDw;
        t.wide = 1;
        t.mt = s.b0 + off / (p.Nh / 2);
        t.nt = off % (p.Nh / 2);
    } else {
        const int blk = s.an + p.Nh;
        const int c = off / blk;
        const int r = off - c * blk;
        if (r < s.an) {
            t.kind = kUnitDz;
            t.nt = s.b0 + c;
            t.mt = s.a0 + r;
        } else {
            t.kind = kUnitDw;
            t.mt = s.b0 + c - s.lag;
            t.nt = r - s.an;
        }
    }
    return t;
}

struct WaveInfo {
    int r0;     // first row of the wave (in the launch's row tensor maps)
    int rows;   // rows of the wave
    int Mt;     // 256-row pair tiles
    int KB_dw;  // 64-deep K blocks of the dW tiles
};

__device__ __forceinline__ WaveInfo wave_info(const BwdParams& p, int w) {
    WaveInfo wi;
    wi.r0 = w * p.chunk;
    wi.rows = min(p.chunk, p.M - wi.r0);
    wi.Mt = (wi.rows + PM - 1) / PM;
    wi.KB_dw = (wi.rows + BK - 1) / BK;
    return wi;
}

// Bounded wait until a device-wide counter reaches `target` (acquire).  Gives
// up when this pair aborts, when another pair has recorded a timeout, or
// after `limit_ns`.
__device__ __forceinline__ bool wait_count(const uint32_t* c, uint32_t target, uint64_t limit_ns,
                                           volatile int* abort_flag, const int* err) {
    if (ld_acquire_gpu_u32(c) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire_gpu_u32(c) >= target) return true;
        if (*abort_flag) return false;
        if (ld_volatile_s32(err) & ERR_TIMEOUT) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------ dZ epilogue

// Per-row constants of dZ = p (K1 + K2 acc) + Bc [column == y], with
// p = 2^(acc s log2e - lse2).  Rows outside the wave and ignored rows get
// lse2 = +inf (p = 0) and no target column, hence a zero dZ row.
struct DzRow {
    long long y;
    float lse2, K1, K2, Bc;
};

__device__ __forceinline__ DzRow dz_row(const BwdParams& p, int grow, bool in_wave) {
    DzRow d{-1, INFINITY, 0.f, 0.f, 0.f};
    if (!in_wave) return d;
    const long long yv = p.y[grow];
    if (yv == p.ignore_index) return d;
    const float lse_v = p.lse[grow];
    const float glp = p.g_lp ? p.g_lp[grow] : 0.f;
    const float gent = (p.ent && p.g_ent) ? p.g_ent[grow] : 0.f;
    const float spz = p.ent ? (lse_v - p.ent_v[grow]) : 0.f;  // sum_j p_j z_j
    const float A = p.scale * gent;
    d.y = yv;
    d.Bc = p.scale * glp;
    d.K1 = A * spz - d.Bc;
    d.K2 = -A * p.scale;
    d.lse2 = lse_v * LOG2E;
    if (yv < 0 || yv >= p.V) atomicOr(p.err, ERR_BAD_TARGET);
    return d;
}

// dZ of 32 columns of this thread's row, from the accumulator columns at
// taddr (vocabulary columns cb, cb + 32), as 16 packed bf16 pairs.  With
// `release`, the accumulator is released after the TMEM read.
__device__ __forceinline__ void dz_words32(uint32_t taddr, int cb, int V, float scale2, const DzRow& d,
                                           bool release, uint32_t tempty, uint32_t (&w)[16]) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr, v);
    tmem_wait_ld();
    if (release) {
        tc_fence_before();
        mbar_arrive_cluster(tempty);
    }
    float dz[32];
    {
        // packed fp32 pairs: p = 2^(acc s log2e - lse2), dz = p (K1 + K2 acc)
        const uint64_t sc2 = f2_pack(scale2, scale2);
        const uint64_t nl = f2_pack(-d.lse2, -d.lse2);
        const uint64_t k1 = f2_pack(d.K1, d.K1), k2 = f2_pack(d.K2, d.K2);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint64_t a = f2_pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            float x0, x1;
            f2_unpack(f2_fma(a, sc2, nl), x0, x1);
            const uint64_t pp = f2_pack(ex2_approx(x0), ex2_approx(x1));
            f2_unpack(f2_mul(pp, f2_fma(a, k2, k1)), dz[2 * j], dz[2 * j + 1]);
        }
    }
    const long long tc = d.y - cb;
    if (tc >= 0 && tc < 32) {
        const uint32_t bit = 1u << static_cast<int>(tc);
#pragma unroll
        for (int j = 0; j < 32; ++j) dz[j] += ((bit >> j) & 1u) ? d.Bc : 0.f;
    }
    const int nv = V - cb;
    if (nv < 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j >= nv) dz[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(dz[2 * j], dz[2 * j + 1]);
}

// One 256-column dZ tile of this thread's row: 4 store boxes of 64 bf16
// columns; the accumulator is released after its last TMEM read.
__device__ __forceinline__ void dz_tile_epilogue(StoreRing& ring, uint8_t* smem, int et, int r,
                                                 uint32_t tbase, int col0, int out_col0, int V,
                                                 float scale2, const DzRow& d, const CUtensorMap* out,
                                                 int out_row, uint32_t tempty) {
#pragma unroll 1
    for (int b = 0; b < BN / 64; ++b) {
        const uint32_t box = store_box_acquire(ring, smem, et);
        uint32_t w[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t wh[16];
            dz_words32(tbase + b * 64 + h * 32, col0 + b * 64 + h * 32, V, scale2, d,
                       b == BN / 64 - 1 && h == 1, tempty, wh);
#pragma unroll
            for (int j = 0; j < 16; ++j) w[h * 16 + j] = wh[j];
        }
        stage_row(box, r, w);
        store_box_release(ring, smem, et, out, out_col0 + b * 64, out_row, false);
    }
}

// One 256-column dX or dW tile of this thread's row: bf16 boxes of 64 columns
// or fp32 boxes of 32 columns, stored or added.
__device__ __forceinline__ void gemm_tile_epilogue(StoreRing& ring, uint8_t* smem, int et, int r,
                                                   uint32_t tbase, bool bf16_out, bool add,
                                                   const CUtensorMap* out, int col0, int row0,
                                                   uint32_t tempty) {
    if (bf16_out) {
#pragma unroll 1
        for (int b = 0; b < BN / 64; ++b) {
            const uint32_t box = store_box_acquire(ring, smem, et);
            uint32_t w[32];
            tmem_row64_to_bf16(tbase + b * 64, w);
            if (b == BN / 64 - 1) {
                tc_fence_before();
                mbar_arrive_cluster(tempty);
            }
            stage_row(box, r, w);
            store_box_release(ring, smem, et, out, col0 + b * 64, row0, false);
        }
    } else {
#pragma unroll 1
        for (int b = 0; b < BN / 32; ++b) {
            const uint32_t box = store_box_acquire(ring, smem, et);
            uint32_t w[32];
            tmem_ld_32x32b_x32(tbase + b * 32, w);
            tmem_wait_ld();
            if (b == BN / 32 - 1) {
                tc_fence_before();
                mbar_arrive_cluster(tempty);
            }
            stage_row(box, r, w);
            store_box_release(ring, smem, et, out, col0 + b * 32, row0, add);
        }
    }
}

// The same through one group's two narrow boxes: 32 bf16 columns per box, or
// 16 fp32 columns per box (two boxes per TMEM load of 32 columns).
__device__ __forceinline__ void gemm_tile_epilogue_narrow(StoreRing& ring, uint8_t* box0, uint32_t bar_id,
                                                          int et, int r, uint32_t tbase, bool bf16_out,
                                                          bool add, const CUtensorMap* out, int col0, int row0,
                                                          uint32_t tempty) {
#pragma unroll 1
    for (int b = 0; b < BN / 32; ++b) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tbase + b * 32, v);
        tmem_wait_ld();
        if (b == BN / 32 - 1) {
            tc_fence_before();
            mbar_arrive_cluster(tempty);
        }
        if (bf16_out) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            narrow_box_store(ring, box0, bar_id, et, r, w, out, col0 + b * 32, row0, false);
        } else {
            narrow_box_store(ring, box0, bar_id, et, r, v, out, col0 + b * 32, row0, add);
            narrow_box_store(ring, box0, bar_id, et, r, v + 16, out, col0 + b * 32 + 16, row0, add);
        }
    }
}

// The kernel is instantiated per set of tile kinds a launch holds, so a
// launch of dZ tiles alone (or of dX and dW tiles alone) carries no code for
// the others.
constexpr int kHasDz = 1, kHasDx = 2, kHasDw = 4;
constexpr int kHasDzWide = 8;  // a launch of wide dZ tiles alone: flp_dz_kernel
constexpr uint32_t DZ_BOX_BYTES = BM * 32 * 2;  // flp_dz_kernel's store box: 128 rows x 32 bf16
static_assert(4 * DZ_BOX_BYTES <= NUM_STG * STG_BYTES, "two boxes per epilogue group");

struct UnitClass {
    bool dz, dx, wide;  // dW when neither dz nor dx; wide: a 256 x 512 dX or dW tile
};

template <int kKinds>
__device__ __forceinline__ UnitClass classify(const BUnit& t) {
    UnitClass c;
    c.dz = (kKinds == kHasDz) || ((kKinds & kHasDz) && t.kind == kUnitDz);
    c.dx = (kKinds == kHasDx) || ((kKinds & kHasDx) && !c.dz && t.kind == kUnitDx);
    c.wide = !c.dz && t.wide != 0;  // wide dZ tiles run in flp_dz_kernel only
    return c;
}

__device__ __forceinline__ int unit_kblocks(const BwdParams& p, const UnitClass& c, const WaveInfo& wi) {
    return c.dz ? p.KB_h : (c.dx ? p.KB_v : wi.KB_dw);
}

// ------------------------------------------------------------------ kernel

// A launch of dX and dW tiles alone (the split and vocabulary-split
// schedules) runs two epilogue groups of four warps (320 threads): group g
// drains every use of accumulator g, so the two halves of a wide tile drain in
// parallel, each through the group's own narrow boxes.  The fused launch keeps
// one group of four warps (192 threads) and 128-byte boxes.
template <int kKinds>
__host__ __device__ constexpr bool two_groups() { return kKinds == (kHasDx | kHasDw); }

template <int kKinds>
__global__ void __launch_bounds__(WIDE_THREADS, 1)
    flp_bwd_kernel(const __grid_constant__ CUtensorMap tmXk,    // X, K-major A of dZ tiles (64 x 128 boxes)
                   const __grid_constant__ CUtensorMap tmWk,    // W, K-major B of dZ tiles (64 x 128)
                   const __grid_constant__ CUtensorMap tmDz,    // dZ buffer: dZ store boxes and K-major A of dX (64 x 128)
                   const __grid_constant__ CUtensorMap tmWmn,   // W, MN-major B of dX (64 x 64)
                   const __grid_constant__ CUtensorMap tmDzMn,  // dZ buffer, MN-major A of dW (64 x 64)
                   const __grid_constant__ CUtensorMap tmXmn,   // X, MN-major B of dW (64 x 64)
                   const __grid_constant__ CUtensorMap tmDx,    // dX store boxes (narrow with two groups)
                   const __grid_constant__ CUtensorMap tmDw,    // dW store / add boxes (narrow with two groups)
                   const __grid_constant__ BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = smem_layout(smem_raw);
    uint8_t* smem = sm.base;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int rofs = static_cast<int>(rank) * BM;  // this CTA's rows / columns inside a pair tile
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmXk);
        tma_prefetch_desc(&tmWk);
        tma_prefetch_desc(&tmDz);
        tma_prefetch_desc(&tmWmn);
        tma_prefetch_desc(&tmDzMn);
        tma_prefetch_desc(&tmXmn);
        tma_prefetch_desc(&tmDx);
        tma_prefetch_desc(&tmDw);
    }
    if (threadIdx.x == 0) griddep_launch_dependents();  // the next launch may be scheduled early
    constexpr bool kTwo = two_groups<kKinds>();
    const uint32_t tmem_base = pair_prologue(sm, warp, 2 + (kTwo ? 4 : 2) * EPI_THREADS);
    griddep_wait();  // the previous launch's results (dZ, the error word) are complete from here on
    const uint64_t limit = p.wait_limit_ns;
    volatile int* abort_flag = sm.abort_flag;

    if (warp == 0) {
        // ------------------------------------------- scheduler + TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t fill_par = 0;  // bit i: parity of the fills of slot i so far
            bool wide_mode = false; // slot layout in use (normal or wide)
            bool ok = true;
            // the leader holds the next ticket one unit ahead, so the global
            // atomic's latency overlaps the current unit's loads
            unsigned long long next_tk = (leader && !p.static_order) ? atomicAdd(p.ticket, 1ull) : 0ull;
            // The leader keeps one unit published ahead of the one it loads, so
            // the peer finds the next unit in its ring when it needs it.
            int published = 0;
            bool ended = false;  // the terminating (-1) unit is in the ring
            for (int it = 0; ok; ++it) {
                const int slot = it % SCHED_SLOTS;
                const uint32_t sph = static_cast<uint32_t>(it / SCHED_SLOTS) & 1u;
                int u;
                if (p.static_order) {
                    u = pair + it * npairs;
                    if (u >= p.total) u = -1;
                } else if (leader) {
                    while (!ended && published < it + 2) {
                        const int ps = published % SCHED_SLOTS;
                        const uint32_t pph = static_cast<uint32_t>(published / SCHED_SLOTS) & 1u;
                        if (!mbar_wait(&sm.sched_empty[ps], pph ^ 1u, limit, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const unsigned long long tk = next_tk - p.ticket_base;
                        const int pu = (tk < static_cast<unsigned long long>(p.total)) ? static_cast<int>(tk) : -1;
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
                const BUnit t = decode_bwd(p, u);
                const UnitClass c = classify<kKinds>(t);
                const WaveInfo wi = wave_info(p, t.wave);
                if (p.deps && !c.dz) {
                    // the dZ tiles this unit reads must be stored first
                    const bool dep_ok =
                        c.dx
                            ? wait_count(p.row_dz + t.mt, 2u * static_cast<uint32_t>(p.Vt) * (t.wave + 1),
                                         limit, abort_flag, p.err)
                            : wait_count(p.col_dz + t.mt,
                                         2u * static_cast<uint32_t>(p.Mt_full * t.wave + wi.Mt), limit,
                                         abort_flag, p.err);
                    if (!dep_ok) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();
                }
                if (c.wide != wide_mode) {
                    // the two slot layouts overlap: every fill of the old one
                    // must have been consumed before the new one is written
                    for (int i = 0; i < STAGES && ok; ++i)
                        ok = mbar_wait(&sm.empty[i], ((fill_par >> i) & 1u) ^ 1u, limit, abort_flag);
                    if (!ok) break;
                    wide_mode = c.wide;
                    stage = 0;
                }
                const int nslots = wide_mode ? STAGES_W : STAGES;
                const int kbn = unit_kblocks(p, c, wi);
                for (int kb = 0; kb < kbn; ++kb) {
                    if (!mbar_wait(&sm.empty[stage], ((fill_par >> stage) & 1u) ^ 1u, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(&sm.full[stage], wide_mode ? PAIR_STAGE_TX_W : PAIR_STAGE_TX);
                    const uint32_t bar = mapa_shared(smem_addr(&sm.full[stage]), 0);
                    uint8_t* a_dst = smem + slot_a(wide_mode, stage);
                    uint8_t* b_dst = smem + slot_b(wide_mode, stage);
                    if (c.dz) {
                        tma_load_2d_pair(a_dst, &tmXk, kb * BK, wi.r0 + t.mt * PM + rofs, bar);
                        tma_load_2d_pair(b_dst, &tmWk, kb * BK, t.nt * BN + rofs, bar);
                    } else if (c.dx) {
                        tma_load_2d_pair(a_dst, &tmDz, kb * BK, t.mt * PM + rofs, bar);  // chunk column kb * BK
                        const int nsub = c.wide ? 2 : 1;
                        for (int h = 0; h < nsub; ++h) {
#pragma unroll
                            for (int j = 0; j < BNH / 64; ++j)
                                tma_load_2d_pair(b_dst + h * B_STAGE_BYTES + j * 8192, &tmWmn,
                                                 (t.nt * nsub + h) * BN + rofs + j * 64, p.vt0 * BN + kb * BK,
                                                 bar);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d_pair(a_dst + j * 8192, &tmDzMn, (t.mt - p.vt0) * PM + rofs + j * 64,
                                             kb * BK, bar);
                        const int nsub = c.wide ? 2 : 1;
                        for (int h = 0; h < nsub; ++h) {
#pragma unroll
                            for (int j = 0; j < BNH / 64; ++j)
                                tma_load_2d_pair(b_dst + h * B_STAGE_BYTES + j * 8192, &tmXmn,
                                                 (t.nt * nsub + h) * BN + rofs + j * 64, wi.r0 + kb * BK, bar);
                        }
                    }
                    fill_par ^= 1u << stage;
                    if (++stage == nslots) stage = 0;
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
            uint32_t full_par = 0;   // bit i: parity of the consumptions of slot i so far
            bool wide_mode = false;  // slot layout in use, switched at the same units as the producer's
            int acc = 0;             // next accumulator (a wide tile takes both, starting here)
            uint32_t tpar = 0;       // bit a: parity of the uses of accumulator a so far
            bool ok = true;
            constexpr uint32_t idesc_kk = idesc_bf16_f32(PM, BN, 0, 0);  // dZ: X and W K-major
            constexpr uint32_t idesc_km = idesc_bf16_f32(PM, BN, 0, 1);  // dX: dZ K-major, W MN-major
            constexpr uint32_t idesc_mm = idesc_bf16_f32(PM, BN, 1, 1);  // dW: dZ^T and X MN-major
            for (int it = 0; ok; ++it) {
                const int slot = it % SCHED_SLOTS;
                const uint32_t sph = static_cast<uint32_t>(it / SCHED_SLOTS) & 1u;
                int u;
                if (p.static_order) {
                    u = pair + it * npairs;
                    if (u >= p.total) break;
                } else {
                    if (!mbar_wait(&sm.sched_full[slot], sph, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    u = sm.sched_val[slot];
                    mbar_arrive(&sm.sched_empty[slot]);
                    if (u < 0) break;
                }
                const BUnit t = decode_bwd(p, u);
                const UnitClass c = classify<kKinds>(t);
                const WaveInfo wi = wave_info(p, t.wave);
                if (c.wide != wide_mode) {
                    wide_mode = c.wide;
                    stage = 0;
                }
                const int nslots = wide_mode ? STAGES_W : STAGES;
                const int kbn = unit_kblocks(p, c, wi);
                // k-block kb of this unit sits in slot (stage + kb) % nslots
                auto wait_full = [&](int kb) {
                    const int s = (stage + kb) % nslots;
                    if (!mbar_wait(&sm.full[s], (full_par >> s) & 1u, limit, abort_flag)) return false;
                    full_par ^= 1u << s;
                    tc_fence_after();
                    return true;
                };
                auto release = [&](int kb) {
                    umma_commit_pair_mc(&sm.empty[(stage + kb) % nslots], PAIR_MASK);  // stage free in both CTAs
                };
                // the MMAs of k-block kb into half h (accumulator acc ^ h; a wide
                // tile's half h reads the B half of its 256-column sub-tile h)
                auto issue = [&](int kb, int h) {
                    const int s = (stage + kb) % nslots;
                    const uint32_t a_base = smem_addr(smem + slot_a(wide_mode, s));
                    const uint32_t b_base = smem_addr(smem + slot_b(wide_mode, s)) + h * B_STAGE_BYTES;
                    const uint32_t d_h = tmem_base + static_cast<uint32_t>((acc ^ h) * BN);
                    if (c.dz) {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            umma_bf16_pair(d_h, operand_desc<0>(a_base, k), operand_desc<0>(b_base, k), idesc_kk,
                                           (kb > 0 || k > 0) ? 1u : 0u);
                    } else if (c.dx) {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            umma_bf16_pair(d_h, operand_desc<0>(a_base, k), operand_desc<1>(b_base, k), idesc_km,
                                           (kb > 0 || k > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            umma_bf16_pair(d_h, operand_desc<1>(a_base, k), operand_desc<1>(b_base, k), idesc_mm,
                                           (kb > 0 || k > 0) ? 1u : 0u);
                    }
                };
                auto wait_tempty = [&](int a) {
                    return mbar_wait(&sm.tempty[a], ((tpar >> a) & 1u) ^ 1u, limit, abort_flag);
                };
                auto publish = [&](int a) {
                    umma_commit_pair_mc(&sm.tfull[a], PAIR_MASK);  // accumulator ready in both CTAs
                    tpar ^= 1u << a;
                };
                if (!c.wide) {
                    if (!wait_tempty(acc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int kb = 0; kb < kbn && ok; ++kb) {
                        ok = wait_full(kb);
                        if (!ok) break;
                        issue(kb, 0);
                        release(kb);
                    }
                    if (!ok) break;
                    publish(acc);
                    acc ^= 1;
                } else {
                    // A wide tile holds both accumulators (half 0 in acc, half 1 in
                    // acc ^ 1), so its first and last STAGES_W k-blocks are issued
                    // half by half: half 0 completes (and is drained) while the
                    // last half-1 MMAs run, and the next tile's half 0 starts while
                    // this tile's half 1 is still drained.
                    const int head = min(STAGES_W, kbn);
                    const int tail0 = max(head, kbn - STAGES_W);
                    if (!wait_tempty(acc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int kb = 0; kb < head && ok; ++kb) {
                        ok = wait_full(kb);
                        if (ok) issue(kb, 0);
                    }
                    if (!ok) break;
                    if (head == kbn) publish(acc);
                    if (!wait_tempty(acc ^ 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int kb = 0; kb < head; ++kb) {
                        issue(kb, 1);
                        release(kb);
                    }
                    for (int kb = head; kb < tail0 && ok; ++kb) {
                        ok = wait_full(kb);
                        if (!ok) break;
                        issue(kb, 0);
                        issue(kb, 1);
                        release(kb);
                    }
                    for (int kb = tail0; kb < kbn && ok; ++kb) {
                        ok = wait_full(kb);
                        if (ok) issue(kb, 0);
                    }
                    if (!ok) break;
                    if (head < kbn) publish(acc);
                    for (int kb = tail0; kb < kbn; ++kb) {
                        issue(kb, 1);
                        release(kb);
                    }
                    publish(acc ^ 1);  // the next tile starts at acc again
                }
                stage = (stage + kbn) % nslots;
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
        const int g = kTwo ? (warp - 2) >> 2 : 0;  // epilogue group (drains accumulator g when kTwo)
        const int et = threadIdx.x - 64 - g * EPI_THREADS;  // 0..127; thread 0 issues the bulk stores
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int r = q * 32 + lane;      // accumulator row == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tempty_leader0 = mapa_shared(smem_addr(&sm.tempty[0]), 0);
        const uint32_t tempty_leader1 = mapa_shared(smem_addr(&sm.tempty[1]), 0);
        const uint32_t bar_box = kTwo ? 1 + 2 * g : 1, bar_vote = kTwo ? 2 + 2 * g : 2;
        uint8_t* nbox0 = smem + SMEM_STG + g * (2 * NBOX_BYTES);  // this group's narrow boxes
        int acc = 0;        // next accumulator (a wide dX tile drains acc, then acc ^ 1)
        uint32_t tpar = 0;  // bit a: parity of the uses of accumulator a so far
        bool ok = true;
        StoreRing ring;
        for (int it = 0;; ++it) {
            const int slot = it % SCHED_SLOTS;
            const uint32_t sph = static_cast<uint32_t>(it / SCHED_SLOTS) & 1u;
            bool got = true;
            int u = -1;
            if (p.static_order) {
                u = pair + it * npairs;
                if (u >= p.total) u = -1;
            } else {
                got = mbar_wait<true>(&sm.sched_full[slot], sph, limit, abort_flag);
                if (got) {
                    u = sm.sched_val[slot];
                    mbar_arrive_cluster(mapa_shared(smem_addr(&sm.sched_empty[slot]), 0));
                }
            }
            BUnit t{};
            UnitClass c{};
            WaveInfo wi{};
            DzRow d{};
            bool ready = got;
            int nacc = 1;
            if (got && u >= 0) {
                t = decode_bwd(p, u);
                c = classify<kKinds>(t);
                wi = wave_info(p, t.wave);
                if (c.dz) {
                    const int lrow = t.mt * PM + rofs + r;  // row inside the wave
                    d = dz_row(p, wi.r0 + lrow, lrow < wi.rows);
                }
                if (p.deps && t.wave > 0 && !c.dx && et == 0) {
                    // a dZ tile overwrites a buffer slot the previous wave's dX
                    // and dW tiles read; a dW tile adds after the previous wave's add
                    const uint32_t tgt_dx = 2u * static_cast<uint32_t>(p.Ndx) * t.wave;
                    const uint32_t tgt_dw = 2u * static_cast<uint32_t>(p.Nh) * t.wave;
                    bool dep_ok;
                    if (c.dz)
                        dep_ok = wait_count(p.dx_done + t.mt, tgt_dx, limit, abort_flag, p.err) &&
                                 wait_count(p.dw_done + t.nt, tgt_dw, limit, abort_flag, p.err);
                    else
                        dep_ok = wait_count(p.dw_done + t.mt, tgt_dw, limit, abort_flag, p.err);
                    if (!dep_ok) raise_abort(sm, p.err);  // the others wait on this thread at the store barriers
                    fence_proxy_async_global();
                }
                nacc = c.wide ? 2 : 1;
                for (int h = 0; h < nacc && ready; ++h) {
                    const int a = acc ^ h;
                    if (kTwo && a != g) continue;  // the other group drains it
                    ready = mbar_wait(&sm.tfull[a], (tpar >> a) & 1u, limit, abort_flag);
                }
            }
            // every epilogue thread of the group takes the same branch (the
            // store barriers below need all of them)
            if (!named_bar_all(bar_vote, EPI_THREADS, ready)) {
                ok = false;
                break;
            }
            if (u < 0) break;
            tc_fence_after();
            for (int h = 0; h < nacc; ++h) {
                const int a = acc ^ h;
                const uint32_t tbase = tmem_base + static_cast<uint32_t>(a * BN) + lane_off;
                const uint32_t tempty = a ? tempty_leader1 : tempty_leader0;
                if constexpr (kTwo) {
                    if (a == g) {
                        if (c.dx)
                            gemm_tile_epilogue_narrow(ring, nbox0, bar_box, et, r, tbase, !p.dx_f32,
                                                      p.dx_add != 0, &tmDx, (t.nt * nacc + h) * BN,
                                                      wi.r0 + t.mt * PM + rofs, tempty);
                        else
                            gemm_tile_epilogue_narrow(ring, nbox0, bar_box, et, r, tbase, p.dw_bf16 != 0,
                                                      t.wave > 0 || p.dw_add0, &tmDw, (t.nt * nacc + h) * BN,
                                                      t.mt * PM + rofs, tempty);
                    }
                } else if (c.dz) {
                    dz_tile_epilogue(ring, smem, et, r, tbase, t.nt * BN, (t.nt - p.vt0) * BN, p.V,
                                     p.scale2, d, &tmDz, t.mt * PM + rofs, tempty);
                } else if (c.dx) {
                    gemm_tile_epilogue(ring, smem, et, r, tbase, !p.dx_f32, p.dx_add != 0, &tmDx,
                                       (t.nt * nacc + h) * BN, wi.r0 + t.mt * PM + rofs, tempty);
                } else {
                    gemm_tile_epilogue(ring, smem, et, r, tbase, p.dw_bf16 != 0, t.wave > 0 || p.dw_add0,
                                       &tmDw, (t.nt * nacc + h) * BN, t.mt * PM + rofs, tempty);
                }
                tpar ^= 1u << a;
            }
            if (p.deps && et == 0 && (c.dz || p.nwaves > 1)) {
                // publish the finished tile: its bulk stores complete, then a release
                bulk_wait_group<0>();
                fence_proxy_async_global();
                if (c.dz) {
                    red_release_gpu_add_u32(p.row_dz + t.mt, 1u);
                    red_release_gpu_add_u32(p.col_dz + t.nt, 1u);
                } else if (c.dx) {
                    red_release_gpu_add_u32(p.dx_done + t.mt, 1u);
                } else {
                    red_release_gpu_add_u32(p.dw_done + t.mt, 1u);
                }
            }
            if (nacc == 1) acc ^= 1;
        }
        if (!ok) {
            raise_abort(sm, p.err);
        }
        if (et == 0) bulk_wait_group<0>();
    }

    pair_epilogue(sm, warp, tmem_base);
}

// ------------------------------------------------------------ wide dZ tiles

// The dZ launch of the split and vocabulary-split schedules (kSegDz2 segments,
// equal tiles with K = H, a static round-robin over the pairs), built like the
// forward: 256 x 512 tiles in both accumulators with the halves staggered at
// the tile ends (wide_tile_mma), and two epilogue groups of four warps, group g
// draining half g into its own store box.  A group computes a box's dZ before
// it waits for that box's previous bulk store to finish reading it.  A half at
// or past the launch's last vocabulary tile (odd tile counts) is computed but
// not stored.  Each half runs the MMAs and the epilogue arithmetic of a
// 256 x 256 dZ tile of flp_bwd_kernel, so both give the same bits.
__global__ void __launch_bounds__(WIDE_THREADS, 1)
    flp_dz_kernel(const __grid_constant__ CUtensorMap tmXk,  // X, K-major A (64 x 128 boxes)
                  const __grid_constant__ CUtensorMap tmWk,  // W, K-major B (64 x 128)
                  const __grid_constant__ CUtensorMap tmDz,  // dZ buffer: store boxes (32 x 128, 64-byte swizzle)
                  const __grid_constant__ BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = smem_layout(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int rofs = static_cast<int>(rank) * BM;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmXk);
        tma_prefetch_desc(&tmWk);
        tma_prefetch_desc(&tmDz);
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
            int issued = 0;
            bool ok = true;
            for (int u = pair; u < p.total && ok; u += npairs) {
                const BUnit t = decode_bwd(p, u);
                const WaveInfo wi = wave_info(p, t.wave);
                for (int kb = 0; kb < p.KB_h; ++kb) {
                    if (p.debug_stop_at > 0 && issued >= p.debug_stop_at - 1) {
                        ok = false;  // injected stall: stop feeding the MMA
                        break;
                    }
                    if (!mbar_wait(&sm.empty[stage], phase ^ 1u, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    load_wide_kblock(sm, stage, leader, &tmXk, wi.r0 + t.mt * PM + rofs, &tmWk,
                                     t.nt * BN + rofs, kb);
                    ++issued;
                    if (++stage == STAGES_W) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && p.debug_stop_at == 0) raise_abort(sm, p.err);
        }
    } else if (warp == 1) {
        // ---------------------------------------------- MMA issuer (leader)
        if (lane == 0 && leader) {
            uint32_t gk = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = pair; u < p.total && ok; u += npairs) {
                ok = wide_tile_mma(sm, tmem_base, gk, acc_phase, p.KB_h, limit, abort_flag);
                acc_phase ^= 1u;
            }
            if (!ok) raise_abort(sm, p.err);
            umma_commit_pair_mc(sm.drain, 0x1);  // every MMA issued so far has completed
            volatile int no_abort = 0;
            mbar_wait(sm.drain, 0, limit, &no_abort);
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int g = (warp - 2) >> 2;                 // the half this group drains
        const int et = threadIdx.x - 64 - g * EPI_THREADS;  // 0..127; thread 0 issues the bulk stores
        const int q = warp & 3;                        // TMEM lane quadrant of this warp
        const int r = q * 32 + lane;                   // accumulator row == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tempty = mapa_shared(smem_addr(&sm.tempty[g]), 0);
        const uint32_t bar_box = 1 + g, bar_vote = 3 + g;  // named barriers of this group
        // two store boxes per group (128 rows x 32 bf16 columns, 64-byte swizzle)
        uint8_t* box_ptr = sm.base + SMEM_STG + g * (2 * DZ_BOX_BYTES);
        uint32_t nbox = 0;  // boxes stored by this group so far; box nbox & 1 is next
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int u = pair; u < p.total; u += npairs) {
            const BUnit t = decode_bwd(p, u);
            const WaveInfo wi = wave_info(p, t.wave);
            const int lrow = t.mt * PM + rofs + r;  // row inside the wave
            const DzRow d = dz_row(p, wi.r0 + lrow, lrow < wi.rows);
            const bool ready = mbar_wait(&sm.tfull[g], acc_phase, limit, abort_flag);
            // every thread of the group takes the same branch (the box barriers need all of them)
            if (!named_bar_all(bar_vote, EPI_THREADS, ready)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int vt = t.nt + g;  // this half's vocabulary tile
            const uint32_t tbase = tmem_base + static_cast<uint32_t>(g * BN) + lane_off;
            if (vt < p.vt_end) {
#pragma unroll 1
                for (int b = 0; b < BN / 32; ++b) {
                    uint32_t w[16];
                    dz_words32(tbase + b * 32, vt * BN + b * 32, p.V, p.scale2, d, b == BN / 32 - 1, tempty, w);
                    // box nbox & 1 was last read by the store two boxes back, which thread 0
                    // waited for before the previous barrier
                    uint8_t* bp = box_ptr + (nbox & 1u) * DZ_BOX_BYTES;
                    const uint32_t row_addr = smem_addr(bp) + r * 64;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_shared_v4(row_addr + ((c ^ ((r >> 1) & 3)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                                     w[4 * c + 3]);
                    fence_proxy_async_smem();
                    if (et == 0) bulk_wait_group_read<0>();  // the other box is free again
                    named_bar_sync(bar_box, EPI_THREADS);
                    if (et == 0) {
                        tma_store_2d(&tmDz, bp, (vt - p.vt0) * BN + b * 32, t.mt * PM + rofs);
                        bulk_commit_group();
                    }
                    ++nbox;
                }
            } else {
                tc_fence_before();
                mbar_arrive_cluster(tempty);
            }
            acc_phase ^= 1u;
        }
        if (!ok) raise_abort(sm, p.err);
        if (et == 0) bulk_wait_group<0>();
    }

    pair_epilogue(sm, warp, tmem_base);
}

}  // namespace flp
