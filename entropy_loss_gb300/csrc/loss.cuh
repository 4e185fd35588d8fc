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
// The kernel also writes d loss / d lp_i, the upstream gradient that
// flp_backward takes.  One block, fixed-order fp64 reductions: deterministic.
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
    if (p.kind == 1) {
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
    const double inv_n = n > 0 ? 1.0 / static_cast<double>(n) : 0.0;
    if (t == 0) *p.loss = static_cast<float>(s_sum[0] * inv_n);
    for (long long i = t; i < p.M; i += LOSS_THREADS) {
        float term = 0.f, g = 0.f;
        if (p.y[i] != p.ignore_index) loss_term(p, i, term, g);
        if (p.per_row) p.per_row[i] = term;
        if (p.grad) p.grad[i] = static_cast<float>(g * inv_n);
    }
}

}  // namespace flp
