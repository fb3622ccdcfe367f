// GRPO clipped-surrogate loss on the selected-token logp path (RL-Kernel
// issue #241, PR 5: ratio, clip, KL, advantage, a declared normaliser and a
// fixed summation order), with its gradient with respect to logp, which is
// the upstream gradient of the fused logp backward.
//
// Per active token t:  r = exp(logp - old),
//   pg = max(-A r, -A clip(r, 1 - eps_lo, 1 + eps_hi)),
//   kl = exp(ref - logp) - (ref - logp) - 1   (when ref is given),
//   l  = pg + beta kl,
//   dl/dlogp = (-A r if the unclipped term is the max, else 0)
//              + beta (1 - exp(ref - logp)).
// Normalisers: 0 token mean (sum l / D), 1 sequence mean of token means,
// 2 sequence mean of token sums; a positive `normalizer` replaces D or the
// number of non-empty sequences.
//
// One CTA of 32 warps.  Segment s (a sequence [cu[s], cu[s+1]), or a chunk of
// 1024 tokens of the single whole-batch sequence when cu is NULL) belongs to
// warp s mod 32; a warp walks its segments in increasing s, its lanes walk a
// segment's tokens with stride 32, and every sum is a fixed xor butterfly over
// the lanes followed by a left fold over the warps in warp order.  The result
// depends only on the inputs and the segment layout, never on timing.
#pragma once

#include "logp_prims.cuh"

namespace flp {

constexpr int kGrpoThreads = 1024;
constexpr int kGrpoWarps = kGrpoThreads / 32;
constexpr int64_t kGrpoChunk = 1024;

struct GrpoArgs {
    const float* logp;
    const float* old_logp;
    const float* ref_logp;      // nullable
    const float* adv;
    const uint8_t* mask;        // nullable
    const int64_t* cu;          // nullable, [nseq + 1]
    int64_t nseq, n;
    int mode;
    float eps_lo, eps_hi, beta, normalizer;
    float* loss;                // [1]
    float* grad;                // [n]
    float* token_loss;          // nullable [n]
};

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// [a, b) of segment s, clamped to [0, n] and made non-decreasing.
__device__ __forceinline__ void grpo_segment(const GrpoArgs& p, int64_t s, int64_t& a, int64_t& b) {
    if (p.cu) {
        a = __ldg(p.cu + s);
        b = __ldg(p.cu + s + 1);
        a = a < 0 ? 0 : (a > p.n ? p.n : a);
        b = b < a ? a : (b > p.n ? p.n : b);
    } else {
        a = s * kGrpoChunk;
        b = a + kGrpoChunk < p.n ? a + kGrpoChunk : p.n;
    }
}

__global__ void __launch_bounds__(kGrpoThreads, 1) k_grpo_loss(GrpoArgs p) {
    __shared__ double sh[kGrpoWarps][4];
    __shared__ double sh_den;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nseg = p.cu ? p.nseq : (p.n + kGrpoChunk - 1) / kGrpoChunk;
    const float lo = 1.f - p.eps_lo, hi = 1.f + p.eps_hi;

    // pass 1: per-token loss and unnormalised gradient, per-segment sums
    double tot = 0.0, cnt = 0.0, seqterm = 0.0, sact = 0.0;
    for (int64_t s = warp; s < nseg; s += kGrpoWarps) {
        int64_t a, b;
        grpo_segment(p, s, a, b);
        double lsum = 0.0, lcnt = 0.0;
        for (int64_t t = a + lane; t < b; t += 32) {
            float l = 0.f, dl = 0.f;
            if (p.mask == nullptr || __ldg(p.mask + t) != 0) {
                const float lp = __ldg(p.logp + t);
                const float A = __ldg(p.adv + t);
                const float r = expf(__fsub_rn(lp, __ldg(p.old_logp + t)));
                const float rc = fminf(fmaxf(r, lo), hi);
                const float p1 = __fmul_rn(-A, r), p2 = __fmul_rn(-A, rc);
                const bool unclipped = p1 >= p2;
                l = unclipped ? p1 : p2;
                dl = unclipped ? p1 : 0.f;
                if (p.ref_logp) {
                    const float d = __fsub_rn(__ldg(p.ref_logp + t), lp);
                    const float e = expf(d);
                    l = __fmaf_rn(p.beta, __fsub_rn(__fsub_rn(e, d), 1.f), l);
                    dl = __fmaf_rn(p.beta, __fsub_rn(1.f, e), dl);
                }
                lsum += (double)l;
                lcnt += 1.0;
            }
            p.grad[t] = dl;
            if (p.token_loss) p.token_loss[t] = l;
        }
        const double ssum = warp_sum_d(lsum), scnt = warp_sum_d(lcnt);
        tot += ssum;
        cnt += scnt;
        if (scnt > 0) {
            sact += 1.0;
            seqterm += (p.mode == 1) ? ssum / scnt : ssum;
        }
    }
    if (lane == 0) {
        sh[warp][0] = tot;
        sh[warp][1] = cnt;
        sh[warp][2] = seqterm;
        sh[warp][3] = sact;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double T = 0.0, C = 0.0, Q = 0.0, A = 0.0;
        for (int w = 0; w < kGrpoWarps; ++w) {
            T += sh[w][0];
            C += sh[w][1];
            Q += sh[w][2];
            A += sh[w][3];
        }
        if (!p.cu) {  // the whole batch is one sequence
            A = C > 0 ? 1.0 : 0.0;
            Q = (p.mode == 1) ? (C > 0 ? T / C : 0.0) : T;
        }
        double den = (p.mode == 0) ? C : A;
        if (p.normalizer > 0.f) den = (double)p.normalizer;
        const double num = (p.mode == 0) ? T : Q;
        p.loss[0] = den > 0 ? __double2float_rn(num / den) : 0.f;
        sh_den = den;
        sh[0][1] = C;   // total active tokens, for the single-sequence weights
    }
    __syncthreads();
    const double den = sh_den, total_cnt = sh[0][1];

    // pass 2: weights
    for (int64_t s = warp; s < nseg; s += kGrpoWarps) {
        int64_t a, b;
        grpo_segment(p, s, a, b);
        double w;
        if (den <= 0) {
            w = 0.0;
        } else if (p.mode == 1) {
            double n_s;
            if (p.cu) {
                double c = 0.0;
                for (int64_t t = a + lane; t < b; t += 32)
                    c += (p.mask == nullptr || __ldg(p.mask + t) != 0) ? 1.0 : 0.0;
                n_s = warp_sum_d(c);
            } else {
                n_s = total_cnt;
            }
            w = n_s > 0 ? 1.0 / (den * n_s) : 0.0;
        } else {
            w = 1.0 / den;
        }
        const float wf = __double2float_rn(w);
        for (int64_t t = a + lane; t < b; t += 32) p.grad[t] = __fmul_rn(p.grad[t], wf);
    }
}

}  // namespace flp
