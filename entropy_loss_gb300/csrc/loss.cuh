// loss.cuh - loss heads on the per-row log-probs of the fused LM head.
//
// The chunked GRPO loss of "Triton MoE improvements and chunked GRPO
// improvements" (section "Chunked Triton GRPO loss") sits on top of the
// lm_head's per-token log-probs.  Two heads, both averaged over the N rows
// whose target is not ignore_index:
//   NLL mean:           term_i = -lp_i
//   clipped surrogate:  r_i = exp(lp_i - old_i),
//                       term_i = -min(r_i A_i, clip(r_i, 1 - eps_low, 1 + eps_high) A_i)
//                                + beta (exp(ref_i - lp_i) - (ref_i - lp_i) - 1)
//   NLL sum:            term_i = -lp_i, not averaged (loss = sum of the terms)
// The kernel also writes d loss / d lp_i, the upstream gradient that
// flp_backward takes.  One block, fixed-order fp64 reductions: deterministic.
//
// flp_policy_loss_kernel generalises the clipped surrogate to sequences (the
// same page's "Setup": loss_type="dapo", importance_sampling_level="sequence",
// num_items_in_batch; "Correctness": grpo / bnpo / dr_grpo / dapo at token
// and sequence level).  Rows [off[b], off[b+1]) are sequence b, n_b its rows
// whose target is not ignore_index, N the sum of the n_b:
//   ratio        token level: log r_t = lp_t - old_t
//                sequence level: log r_t = (1/n_b) sum_{u in b} (lp_u - old_u)
//   term_t       -min(r_t A_t, clip(r_t, 1 - eps_low, 1 + eps_high) A_t) + beta kl_t
//   aggregation  token mean (bnpo): 1/N; sequence mean (grpo): 1/(B max(n_b, 1))
//                per token of b; sum over a normaliser (dapo: num_items_in_batch,
//                dr_grpo: B x the longest completion): 1/D, D <= 0 -> N
// A sequence-level ratio makes every term of b depend on every lp_u of b:
// d loss / d lp_u = (1/n_b) sum_{t in b} c_t d term_t / d log r_b + c_u d kl_u / d lp_u.
#pragma once
#include <cstdint>

namespace flp {

constexpr int LOSS_THREADS = 1024;

struct LossParams {
    const float* lp;
    const long long* y;
    long long M;
    long long ignore_index;
    int kind;  // 1: NLL mean, 2: clipped surrogate
    const float* old_lp;
    const float* adv;
    const float* ref_lp;  // may be null (no KL term)
    float eps_low, eps_high, beta;
    float* per_row;  // may be null
    float* grad;     // may be null
    float* loss;
};

// Per-row loss term and its derivative with respect to lp_i (before the 1/N).
__device__ __forceinline__ void loss_term(const LossParams& p, long long i, float& term, float& g) {
    const float lp = p.lp[i];
    if (p.kind == 1 || p.kind == 3) {
        term = -lp;
        g = -1.f;
        return;
    }
    const float a = p.adv[i];
    const float r = expf(lp - p.old_lp[i]);
    const float rc = fminf(fmaxf(r, 1.f - p.eps_low), 1.f + p.eps_high);
    const float s1 = r * a, s2 = rc * a;
    const bool unclipped = s1 <= s2;
    term = -(unclipped ? s1 : s2);
    g = unclipped ? -s1 : 0.f;
    if (p.ref_lp && p.beta != 0.f) {
        const float d = p.ref_lp[i] - lp;
        const float ed = expf(d);
        term += p.beta * (ed - d - 1.f);
        g += p.beta * (1.f - ed);
    }
}

__global__ void __launch_bounds__(LOSS_THREADS) flp_loss_kernel(const LossParams p) {
    __shared__ double s_sum[LOSS_THREADS];
    __shared__ long long s_cnt[LOSS_THREADS];
    const int t = threadIdx.x;
    double sum = 0.0;
    long long cnt = 0;
    for (long long i = t; i < p.M; i += LOSS_THREADS) {
        if (p.y[i] == p.ignore_index) continue;
        float term, g;
        loss_term(p, i, term, g);
        sum += static_cast<double>(term);
        ++cnt;
    }
    s_sum[t] = sum;
    s_cnt[t] = cnt;
    __syncthreads();
    for (int w = LOSS_THREADS / 2; w > 0; w >>= 1) {  // fixed pairing order
        if (t < w) {
            s_sum[t] += s_sum[t + w];
            s_cnt[t] += s_cnt[t + w];
        }
        __syncthreads();
    }
    const long long n = s_cnt[0];
    // kind 3 sums the terms; the others average them over the N valid rows
    const double inv_n = p.kind == 3 ? 1.0 : (n > 0 ? 1.0 / static_cast<double>(n) : 0.0);
    if (t == 0) *p.loss = static_cast<float>(s_sum[0] * inv_n);
    for (long long i = t; i < p.M; i += LOSS_THREADS) {
        float term = 0.f, g = 0.f;
        if (p.y[i] != p.ignore_index) loss_term(p, i, term, g);
        if (p.per_row) p.per_row[i] = term;
        if (p.grad) p.grad[i] = static_cast<float>(g * inv_n);
    }
}

struct PolicyLossParams {
    const float* lp;
    const long long* y;
    long long M;
    long long ignore_index;
    const long long* off;  // [B + 1] row offsets of the sequences; null: one sequence of all rows
    long long B;
    const float* old_lp;
    const float* adv;
    const float* ref_lp;  // may be null (no KL term)
    double eps_low, eps_high, beta;
    int is_level;     // 0: token-level ratio, 1: sequence-level ratio
    int aggregation;  // 0: token mean, 1: sequence mean, 2: sum over the normaliser
    double normalizer;
    float* per_row;  // may be null
    float* grad;     // may be null
    float* loss;
};

// Rows [r0, r1) of sequence b, clamped to [0, M) (an inverted range is empty).
__device__ __forceinline__ void seq_rows(const PolicyLossParams& p, long long b, long long& r0,
                                         long long& r1) {
    if (!p.off) {
        r0 = 0;
        r1 = p.M;
        return;
    }
    r0 = min(max(p.off[b], 0ll), p.M);
    r1 = min(max(p.off[b + 1], r0), p.M);
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ long long warp_sum(long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One block: warp w takes sequences w, w + 32, ...; every sum runs in a fixed
// order (lane-strided rows, then a fixed butterfly), so results are
// deterministic.  All arithmetic in fp64, so the clip decisions are taken in
// the precision of the definition.
__global__ void __launch_bounds__(LOSS_THREADS) flp_policy_loss_kernel(const PolicyLossParams p) {
    constexpr int WARPS = LOSS_THREADS / 32;
    __shared__ double s_loss[WARPS];
    __shared__ long long s_cnt[WARPS];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const long long B = p.off ? p.B : 1;
    // rows outside every sequence and ignored rows: zero term and gradient
    for (long long i = t; i < p.M; i += LOSS_THREADS) {
        if (p.per_row) p.per_row[i] = 0.f;
        if (p.grad) p.grad[i] = 0.f;
    }
    long long cnt = 0;
    for (long long b = warp; b < B; b += WARPS) {
        long long r0, r1;
        seq_rows(p, b, r0, r1);
        for (long long i = r0 + lane; i < r1; i += 32) cnt += (p.y[i] != p.ignore_index) ? 1 : 0;
    }
    cnt = warp_sum(cnt);
    if (lane == 0) s_cnt[warp] = cnt;
    __syncthreads();  // also orders the zero fill before the writes below
    long long N = 0;
    for (int w = 0; w < WARPS; ++w) N += s_cnt[w];
    const double D = (p.aggregation == 2 && p.normalizer > 0.0) ? p.normalizer : static_cast<double>(N);
    const double lo = 1.0 - p.eps_low, hi = 1.0 + p.eps_high;
    double wloss = 0.0;
    for (long long b = warp; b < B; b += WARPS) {
        long long r0, r1;
        seq_rows(p, b, r0, r1);
        double sl = 0.0;
        long long nb = 0;
        for (long long i = r0 + lane; i < r1; i += 32) {
            if (p.y[i] == p.ignore_index) continue;
            sl += static_cast<double>(p.lp[i]) - static_cast<double>(p.old_lp[i]);
            ++nb;
        }
        sl = warp_sum(sl);
        nb = warp_sum(nb);
        const double seq_log_r = nb > 0 ? sl / static_cast<double>(nb) : 0.0;
        const double c = p.aggregation == 0   ? (N > 0 ? 1.0 / static_cast<double>(N) : 0.0)
                         : p.aggregation == 1 ? 1.0 / (static_cast<double>(B) * static_cast<double>(nb > 0 ? nb : 1))
                                              : (D > 0.0 ? 1.0 / D : 0.0);
        double lsum = 0.0, G = 0.0;
        for (long long i = r0 + lane; i < r1; i += 32) {
            if (p.y[i] == p.ignore_index) continue;
            const double lp = p.lp[i];
            const double a = p.adv[i];
            const double log_r = p.is_level == 1 ? seq_log_r : lp - static_cast<double>(p.old_lp[i]);
            const double r = exp(log_r);
            const double rc = fmin(fmax(r, lo), hi);
            const double s1 = r * a, s2 = rc * a;
            const bool unclipped = s1 <= s2;
            double term = -(unclipped ? s1 : s2);
            const double dterm = unclipped ? -s1 : 0.0;  // d term / d log r
            double gkl = 0.0;
            if (p.ref_lp && p.beta != 0.0) {
                const double d = static_cast<double>(p.ref_lp[i]) - lp;
                const double ed = exp(d);
                term += p.beta * (ed - d - 1.0);
                gkl = p.beta * (1.0 - ed);
            }
            lsum += term;
            if (p.per_row) p.per_row[i] = static_cast<float>(term);
            if (p.is_level == 1) {
                G += dterm;
                if (p.grad) p.grad[i] = static_cast<float>(c * gkl);  // completed below
            } else if (p.grad) {
                p.grad[i] = static_cast<float>(c * (dterm + gkl));
            }
        }
        lsum = warp_sum(lsum);
        wloss += c * lsum;
        if (p.is_level == 1 && p.grad && nb > 0) {
            G = warp_sum(G);
            const double gs = c * G / static_cast<double>(nb);
            for (long long i = r0 + lane; i < r1; i += 32) {  // the rows this lane wrote above
                if (p.y[i] == p.ignore_index) continue;
                const double lp = p.lp[i];
                double gkl = 0.0;
                if (p.ref_lp && p.beta != 0.0) gkl = p.beta * (1.0 - exp(static_cast<double>(p.ref_lp[i]) - lp));
                p.grad[i] = static_cast<float>(c * gkl + gs);
            }
        }
    }
    if (lane == 0) s_loss[warp] = wloss;
    __syncthreads();
    if (t == 0) {
        double total = 0.0;
        for (int w = 0; w < WARPS; ++w) total += s_loss[w];
        *p.loss = static_cast<float>(total);
    }
}

}  // namespace flp
