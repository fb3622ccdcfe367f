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
// number of non-empty sequences.  Tokens outside every sequence count as
// inactive (l = 0, gradient 0).
//
// The batch is cut into fixed chunks of 256 tokens (one warp each),
// independent of the sequence layout, so the work per warp is the same
// whatever the sequence lengths:
//   1. k_grpo_terms: each warp takes a contiguous range of chunks.  It loads
//      a chunk (8 tokens per lane in two groups of 4, 16-byte accesses when
//      the arrays allow) and finds the sequences that cross it (for its first
//      chunk a 32-ary search over cu_seqlens, later resuming at the last
//      sequence seen; overlapped with the loads).  For each such run
//      (sequence s within chunk w) it sums l and counts the active tokens;
//      the run's sums go to piece slot s + w (slots of distinct runs never
//      collide: a later sequence only meets later chunks).  Each token's
//      unnormalised gradient (or, when the weight is uniform and known up
//      front, the final one) and loss are written, with the chunk's loss
//      sum, active count and first sequence;
//   2. k_grpo_reduce: G CTAs (G fixed by the shape) each fold a
//      fixed share of the chunk totals and of the sequences (each sequence's
//      pieces give its active count and mean); the CTA that finishes last
//      folds the G partials in order into the loss and the weight;
//   3. k_grpo_scale (when the weight was not known up front): each token's
//      gradient, kept in L2 by pass 1, times its sequence's weight.
// Within a 256-token chunk the sums are plain FP32 (each lane's 8 tokens in
// order, then the xor butterfly: an error of at most about 12 u times the
// chunk's sum of |l|); from the chunk level up they are two-float (hi + lo)
// compensated sums in FP32 (Knuth's TwoSum per addition; the pair carries
// about 44 significant bits), so the error does not grow with the batch: the
// FP64 unit of this GPU is far too slow to accumulate per token.  Token
// counts are integers.  Every fold has an order fixed by the token positions
// and the sequence layout, never by the grid or by timing.
#pragma once

#include "logp_prims.cuh"

namespace flp {

constexpr int kGrpoPassThreads = 256;                                // token passes: 8 warps per CTA
constexpr int kGrpoLaneTokens = 8;
constexpr int64_t kGrpoChunk = 32 * kGrpoLaneTokens;                 // 256 tokens per warp

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
    float prescale;             // > 0: the uniform weight, applied by pass 1 (no pass 4)
    float* loss;                // [1]
    float* grad;                // [n]
    float* token_loss;          // nullable [n]
};

// Two-float sum: value = hi + lo.
struct FF {
    float hi, lo;
};

// Knuth's TwoSum: s + e == a + b exactly (s = fl(a + b)).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ FF ff_add(FF x, float y) {
    float s, e;
    two_sum(x.hi, y, s, e);
    return {s, __fadd_rn(x.lo, e)};
}
__device__ __forceinline__ FF ff_add(FF x, FF y) {
    float s, e;
    two_sum(x.hi, y.hi, s, e);
    return {s, __fadd_rn(__fadd_rn(x.lo, y.lo), e)};
}
// Lane 0 holds the sum over the warp (fixed xor butterfly).
__device__ __forceinline__ FF ff_warp_sum(FF v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const FF o{__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)};
        v = ff_add(v, o);
    }
    return v;
}
// An infinite or NaN hi makes lo meaningless (inf - inf): keep hi alone.
__device__ __forceinline__ double ff_value(FF v) {
    return isfinite(v.hi) ? (double)v.hi + (double)v.lo : (double)v.hi;
}
__device__ __forceinline__ int64_t warp_sum_i64(int64_t v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// The fold's first level has G CTAs, G a function of the shape only (so
// the fold order is fixed by the layout): max(sequences, chunks) / 256
// rounded up, at least 1 and at most 1024.
constexpr int kGrpoFoldMaxCtas = 1024;
constexpr int kGrpoReduceThreads = 256;

// e^x as 2^(x log2 e), the power of two from the special-function unit
// (ex2.approx, flushing subnormal results to 0): within a few ulp for
// |x| <~ 1, the error growing by about |x| 2^-24 from rounding x log2 e.
__device__ __forceinline__ float grpo_exp(float x) { return ex2_ftz(__fmul_rn(x, 1.4426950408889634f)); }

struct GrpoWork {
    double* den;          // [2]: the normaliser, the number of active tokens
    float* wt;            // [1]: the uniform weight (token mean, sequence mean of sums, or one sequence)
    unsigned* ticket;     // [1]: CTAs of the fold that are done (zeroed by pass 1, reset by the last CTA)
    FF* part_t;           // [kGrpoFoldMaxCtas]: per fold CTA, loss sum
    FF* part_q;           //   sum of sequence means
    int64_t* part_c;      //   active tokens
    int64_t* part_a;      //   sequences with an active token
    FF* chunk_sum;        // [nchunks]: loss sum of each 256-token chunk
    int64_t* chunk_cnt;   // [nchunks]: its active tokens
    FF* piece;            // [nseq + nchunks]: loss sum of sequence s within chunk w, at s + w
    int64_t* piece_cnt;
    int64_t* chunk_first; // [nchunks]: the first sequence that may meet each chunk
    float* seg_inv;       // [nseq]: 1 / (active tokens of each sequence), 0 for none
};

__device__ __forceinline__ int64_t grpo_chunks(int64_t n) { return (n + kGrpoChunk - 1) / kGrpoChunk; }

// cu_seqlens[s] clamped to [0, n].
__device__ __forceinline__ int64_t grpo_cu(const GrpoArgs& p, int64_t s) {
    const int64_t v = __ldg(p.cu + s);
    return v < 0 ? 0 : (v > p.n ? p.n : v);
}

// The largest s in [0, nseq] with cu[s] <= x, or -1: a 32-ary search by the
// whole warp (each step probes the last entry of 32 equal blocks and keeps
// the first block whose last entry is above x).  All lanes must call it.
__device__ __forceinline__ int64_t grpo_find(const GrpoArgs& p, int64_t x, int lane) {
    int lo = 0, hi = (int)p.nseq + 1;   // entries before lo are <= x; [lo, hi) undecided (nseq < 2^31 - 1)
    while (lo < hi) {
        const int step = (hi - lo + 31) >> 5;
        const int first = lo + lane * step;
        const int end = min(first + step, hi);
        const bool le = first < hi && grpo_cu(p, end - 1) <= x;
        const int k = __popc(__ballot_sync(0xffffffffu, le));
        const int nlo = min(lo + k * step, hi);
        hi = nlo < hi ? min(lo + (k + 1) * step, hi) - 1 : hi;   // block k's last entry is above x
        lo = nlo;
    }
    return (int64_t)lo - 1;
}

// The sequences that meet the chunk starting at token c0: the first one
// (found by the search, or recorded by pass 1) and the next 32 boundaries,
// fetched by the lanes as chunk-local offsets clamped to [0, 256].  Taken
// before the chunk's tokens are used, so that these L2 round trips overlap
// the tokens' loads from HBM.
struct GrpoRuns {
    int64_t s;     // the first sequence that may meet the chunk
    int bnd;       // lane j: cu[s + j] - c0 clamped to [0, 256] (256 past cu[nseq])
    float aux;     // lane j: aux[s + j] when an aux array is given (s + j < nseq), else 0
};

__device__ __forceinline__ GrpoRuns grpo_runs_at(const GrpoArgs& p, int64_t s, int64_t c0, int lane,
                                                 const float* aux) {
    GrpoRuns r{s < 0 ? 0 : s, (int)kGrpoChunk, 0.f};
    const int64_t idx = r.s + lane;
    if (idx <= p.nseq) {
        const int64_t d = grpo_cu(p, idx) - c0;
        r.bnd = d < 0 ? 0 : (d > kGrpoChunk ? (int)kGrpoChunk : (int)d);
    }
    if (aux && idx < p.nseq) r.aux = aux[idx];
    return r;
}
__device__ __forceinline__ GrpoRuns grpo_runs_begin(const GrpoArgs& p, int64_t c0, int lane) {
    if (p.cu == nullptr) return GrpoRuns{0, 0, 0.f};
    return grpo_runs_at(p, grpo_find(p, c0, lane), c0, lane, nullptr);
}

// Calls f(s, ua, ub, aux_s) for each sequence s whose tokens meet the chunk
// of nv tokens from c0, in sequence order, with [ua, ub) the chunk-local
// indices of its tokens there (never empty).  Warp-uniform; boundaries are
// fetched 32 at a time.  kAux: pass the aux value (else 0, no shuffle).
template <bool kAux, class F>
__device__ __forceinline__ void grpo_runs(const GrpoArgs& p, GrpoRuns r, int64_t c0, int nv, int lane,
                                          const float* aux, F&& f) {
    if (p.cu == nullptr) {
        f((int64_t)0, 0, nv, 0.f);   // one sequence: the whole batch
        return;
    }
    if (r.s < p.nseq) {   // the common case: the chunk lies inside sequence r.s
        const int a0 = __shfl_sync(0xffffffffu, r.bnd, 0), b0 = __shfl_sync(0xffffffffu, r.bnd, 1);
        if (a0 == 0 && b0 >= nv) {
            f(r.s, 0, nv, kAux ? __shfl_sync(0xffffffffu, r.aux, 0) : 0.f);
            return;
        }
    }
    while (r.s < p.nseq) {
        for (int j = 0; j < 31; ++j) {
            const int a = __shfl_sync(0xffffffffu, r.bnd, j);
            if (r.s + j >= p.nseq || a >= nv) return;
            const int b = min(__shfl_sync(0xffffffffu, r.bnd, j + 1), nv);
            const float x = kAux ? __shfl_sync(0xffffffffu, r.aux, j) : 0.f;
            if (a < b) f(r.s + j, a, b, x);
        }
        r = grpo_runs_at(p, r.s + 31, c0, lane, aux);
    }
}

// Programmatic dependent launch: the fold and the scale pass are launched
// while their predecessor runs and wait here (griddepcontrol.wait returns
// once the previous grid has completed and its memory is visible; without
// the launch attribute it returns at once).  A predecessor lets them launch
// as soon as each of its CTAs has started.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// L2 eviction policies (createpolicy): inputs are streamed once and leave
// L2 first; unscaled gradients that the scale pass re-reads stay longest.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ float4 ld_f4_hint(const float* p, uint64_t pol) {
    float4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ float4 ld_f4_hint_rw(const float* p, uint64_t pol) {   // memory this kernel writes
    float4 v;
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p), "l"(pol)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_f4_hint(float* p, float4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ uint32_t ld_u32_hint(const void* p, uint64_t pol) {
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
    return v;
}

// Token layout of a chunk: lane L holds tokens u = 128 i + 4 L + e (i < 2,
// e < 4) at index q = 4 i + e, so each 16-byte access of the warp covers 512
// contiguous bytes.  kVec: the arrays are 16-byte aligned (the mask 4-byte),
// whole groups of 4 use vector accesses; otherwise every access is scalar.
// kRw: the array is written by the same kernel (no read-only path).
template <bool kVec, bool kRw = false>
__device__ __forceinline__ void grpo_ld8(const float* base, int lane, int nvalid, float (&v)[kGrpoLaneTokens],
                                         uint64_t pol) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int u = 128 * i + 4 * lane;
        if (kVec && u + 4 <= nvalid) {
            const float4 x = kRw ? ld_f4_hint_rw(base + u, pol) : ld_f4_hint(base + u, pol);
            v[4 * i] = x.x;
            v[4 * i + 1] = x.y;
            v[4 * i + 2] = x.z;
            v[4 * i + 3] = x.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[4 * i + e] = u + e < nvalid ? (kRw ? base[u + e] : __ldg(base + u + e)) : 0.f;
        }
    }
}
template <bool kVec>
__device__ __forceinline__ void grpo_st8(float* base, int lane, int nvalid, const float (&v)[kGrpoLaneTokens],
                                         uint64_t pol) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int u = 128 * i + 4 * lane;
        if (kVec && u + 4 <= nvalid) {
            st_f4_hint(base + u, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]), pol);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (u + e < nvalid) base[u + e] = v[4 * i + e];
        }
    }
}
// Bit q set: token q of the lane exists (u < nvalid) and its mask byte is
// nonzero.  Both groups' mask words are loaded before either is decoded.
template <bool kVec>
__device__ __forceinline__ uint32_t grpo_active8(const uint8_t* mask, int lane, int nvalid, uint64_t pol) {
    const int u0 = 4 * lane, u1 = 128 + 4 * lane;
    if (mask == nullptr) {
        uint32_t act = 0;
#pragma unroll
        for (int q = 0; q < kGrpoLaneTokens; ++q)
            if ((q < 4 ? u0 : u1) + (q & 3) < nvalid) act |= 1u << q;
        return act;
    }
    if (kVec && u1 + 4 <= nvalid) {   // both groups whole (every group of a full chunk)
        const uint32_t m0 = ld_u32_hint(mask + u0, pol), m1 = ld_u32_hint(mask + u1, pol);
        // bytes != 0 -> 1 in each byte, then the four bits gathered by a multiply
        const uint32_t b0 = __vcmpne4(m0, 0u) & 0x01010101u, b1 = __vcmpne4(m1, 0u) & 0x01010101u;
        return ((b0 * 0x01020408u) >> 24) | (((b1 * 0x01020408u) >> 24) << 4);
    }
    uint8_t m[kGrpoLaneTokens];
#pragma unroll
    for (int q = 0; q < kGrpoLaneTokens; ++q) {
        const int u = (q < 4 ? u0 : u1) + (q & 3);
        m[q] = u < nvalid ? __ldg(mask + u) : 0;
    }
    uint32_t act = 0;
#pragma unroll
    for (int q = 0; q < kGrpoLaneTokens; ++q)
        if (m[q] != 0) act |= 1u << q;
    return act;
}

// Bits of the lane's tokens with chunk index u in [ua, ub).
__device__ __forceinline__ uint32_t grpo_in8(int lane, int ua, int ub) {
    uint32_t in = 0;
#pragma unroll
    for (int q = 0; q < kGrpoLaneTokens; ++q) {
        const int u = 128 * (q >> 2) + 4 * lane + (q & 3);
        if (u >= ua && u < ub) in |= 1u << q;
    }
    return in;
}

template <bool kVec>
__global__ void __launch_bounds__(kGrpoPassThreads, 4) k_grpo_terms(GrpoArgs p, GrpoWork wk) {
    const int lane = threadIdx.x & 31;
    const int64_t nchunks = grpo_chunks(p.n);
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const float clo = 1.f - p.eps_lo, chi = 1.f + p.eps_hi;
    griddep_launch_dependents();
    const uint64_t in_pol = l2_evict_first();
    // the scale pass re-reads the gradients: keep them in L2 (else they are final)
    const uint64_t g_pol = p.prescale > 0.f ? l2_evict_first() : l2_evict_last();
    if (blockIdx.x == 0 && threadIdx.x == 0) *wk.ticket = 0u;
    // each warp takes a contiguous range of chunks: only its first chunk needs
    // the search, later ones resume the run walk at the last sequence seen
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t w_end = (gw + 1) * nchunks / nwarps;
    int64_t s_resume = -1;
    for (int64_t w = gw * nchunks / nwarps; w < w_end; ++w) {
        const int64_t c0 = w * kGrpoChunk;
        const int nv = (int)(p.n - c0 < kGrpoChunk ? p.n - c0 : kGrpoChunk);   // tokens in the chunk
        float lp[kGrpoLaneTokens], od[kGrpoLaneTokens], av[kGrpoLaneTokens], rf[kGrpoLaneTokens];
        grpo_ld8<kVec>(p.logp + c0, lane, nv, lp, in_pol);
        grpo_ld8<kVec>(p.old_logp + c0, lane, nv, od, in_pol);
        grpo_ld8<kVec>(p.adv + c0, lane, nv, av, in_pol);
        if (p.ref_logp) grpo_ld8<kVec>(p.ref_logp + c0, lane, nv, rf, in_pol);
        const uint32_t act = grpo_active8<kVec>(p.mask ? p.mask + c0 : nullptr, lane, nv, in_pol);
        // overlaps the loads above
        const GrpoRuns runs = (s_resume < 0 || p.cu == nullptr) ? grpo_runs_begin(p, c0, lane)
                                                                 : grpo_runs_at(p, s_resume, c0, lane, nullptr);
        int64_t s_last = runs.s;
        if (p.cu && p.mode == 1 && lane == 0) wk.chunk_first[w] = runs.s;
        float l[kGrpoLaneTokens], dl[kGrpoLaneTokens];
#pragma unroll
        for (int q = 0; q < kGrpoLaneTokens; ++q) {
            const float r = grpo_exp(__fsub_rn(lp[q], od[q]));
            const float rc = fminf(fmaxf(r, clo), chi);
            const float p1 = __fmul_rn(-av[q], r), p2 = __fmul_rn(-av[q], rc);
            const bool unclipped = p1 >= p2;
            l[q] = unclipped ? p1 : p2;
            dl[q] = unclipped ? p1 : 0.f;
            if (p.ref_logp) {
                const float d = __fsub_rn(rf[q], lp[q]);
                const float e = grpo_exp(d);
                l[q] = __fmaf_rn(p.beta, __fsub_rn(__fsub_rn(e, d), 1.f), l[q]);
                dl[q] = __fmaf_rn(p.beta, __fsub_rn(1.f, e), dl[q]);
            }
            // inactive tokens: 0 (their inputs may be anything)
            const bool on = (act >> q) & 1u;
            l[q] = on ? l[q] : 0.f;
            dl[q] = on ? dl[q] : 0.f;
        }
        FF tot{0.f, 0.f};
        int64_t tcnt = 0;
        uint32_t inseq = 0;
        grpo_runs<false>(p, runs, c0, nv, lane, nullptr, [&](int64_t s, int ua, int ub, float) {
            s_last = s;
            // within the chunk, plain FP32: the lane's tokens in order, then the
            // xor butterfly (lane 0 holds the result)
            float rs = 0.f;
            uint32_t in;
            if (ua == 0 && ub == nv) {   // the whole chunk: no membership tests
                in = 0xffu;
#pragma unroll
                for (int q = 0; q < kGrpoLaneTokens; ++q) rs = __fadd_rn(rs, l[q]);
            } else {
                in = grpo_in8(lane, ua, ub);
#pragma unroll
                for (int q = 0; q < kGrpoLaneTokens; ++q) rs = __fadd_rn(rs, ((in >> q) & 1u) ? l[q] : 0.f);
            }
            inseq |= in;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) rs = __fadd_rn(rs, __shfl_xor_sync(0xffffffffu, rs, off));
            const int cnt = __reduce_add_sync(0xffffffffu, __popc(in & act));
            if (p.cu && p.mode != 0 && lane == 0) {
                wk.piece[s + w] = FF{rs, 0.f};
                wk.piece_cnt[s + w] = cnt;
            }
            tot = ff_add(tot, rs);
            tcnt += cnt;
        });
        if (p.cu && inseq != 0xffu) {   // tokens outside every sequence
#pragma unroll
            for (int q = 0; q < kGrpoLaneTokens; ++q) {
                const bool in = (inseq >> q) & 1u;
                l[q] = in ? l[q] : 0.f;
                dl[q] = in ? dl[q] : 0.f;
            }
        }
        if (p.prescale > 0.f) {
#pragma unroll
            for (int q = 0; q < kGrpoLaneTokens; ++q) dl[q] = __fmul_rn(dl[q], p.prescale);
        }
        grpo_st8<kVec>(p.grad + c0, lane, nv, dl, g_pol);
        if (p.token_loss) grpo_st8<kVec>(p.token_loss + c0, lane, nv, l, in_pol);
        if (lane == 0) {
            wk.chunk_sum[w] = tot;
            wk.chunk_cnt[w] = tcnt;
        }
        s_resume = s_last;   // no later chunk meets an earlier sequence
    }
}

// The mean of a sequence as two floats: sum / cnt, with the remainder of the
// high quotient carried into the low part.
__device__ __forceinline__ FF ff_div_count(FF s, int64_t cnt) {
    const float c = (float)cnt;
    const float q = __fdiv_rn(s.hi, c);
    const float r = __fmaf_rn(-q, c, s.hi);   // s.hi - q c, exact for a correctly rounded q (c < 2^24)
    return {q, __fdiv_rn(__fadd_rn(r, s.lo), c)};
}

// Folds v over the CTA: the fixed butterfly in each warp, then warp order
// (thread 0 gets the result; every thread must call it).
template <int kWarps>
__device__ __forceinline__ FF cta_fold(FF v, int64_t& c, FF* sh_v, int64_t* sh_c) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = ff_warp_sum(v);
    c = warp_sum_i64(c);
    __syncthreads();   // the shared slots may still be read by a previous fold
    if (lane == 0) {
        sh_v[warp] = v;
        sh_c[warp] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        v = FF{0.f, 0.f};
        c = 0;
        for (int w = 0; w < kWarps; ++w) {
            v = ff_add(v, sh_v[w]);
            c += sh_c[w];
        }
    }
    return v;
}

constexpr int64_t kGrpoLongPieces = 64;   // sequences with more pieces are folded by a whole warp

// The fold of the loss and the normaliser, G CTAs (1 when n == 0).  CTA b
// takes the b-th equal share of the chunk totals and, for the sequence
// normalisers, of the sequences: one lane per sequence folds up to 64 of its
// chunk pieces (chunks floor(a / 256) .. floor((b - 1) / 256), at slots
// s + chunk) in piece order; a longer sequence is folded by its whole warp
// (lane-strided, fixed butterfly) -- which of the two depends only on the
// sequence -- giving its active count (kept for the scale pass) and mean.
// Each CTA writes its partials; the CTA that finishes last (an atomic
// ticket, no waiting) folds the partials in CTA order and writes the loss,
// the normaliser and the uniform weight.
__global__ void __launch_bounds__(kGrpoReduceThreads) k_grpo_reduce(GrpoArgs p, GrpoWork wk) {
    constexpr int kW = kGrpoReduceThreads / 32;
    __shared__ FF sh_v[kW];
    __shared__ int64_t sh_c[kW];
    __shared__ bool last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int64_t nchunks = grpo_chunks(p.n);
    const bool seqs = p.cu != nullptr && p.mode != 0 && p.n > 0;
    griddep_launch_dependents();
    // cu_seqlens is the caller's: its first bounds are read before the wait
    const int64_t qs = seqs ? (p.nseq + G - 1) / G : 0;
    const int64_t s0 = b * qs, s1 = seqs ? (s0 + qs < p.nseq ? s0 + qs : p.nseq) : 0;
    int64_t a_first = 0, e_first = 0;
    if (s0 + 32 * warp + lane < s1) {
        a_first = grpo_cu(p, s0 + 32 * warp + lane);
        e_first = grpo_cu(p, s0 + 32 * warp + lane + 1);
    }
    griddep_wait();
    // chunk totals [b ps, (b + 1) ps): the thread's first one is loaded now,
    // with the sequences' first pieces below, and added first
    const int64_t ps = (nchunks + G - 1) / G;
    const int64_t k1 = (b + 1) * ps < nchunks ? (b + 1) * ps : nchunks;
    const int64_t kf = b * ps + threadIdx.x;
    const FF t_first = kf < k1 ? wk.chunk_sum[kf] : FF{0.f, 0.f};
    const int64_t c_first = kf < k1 ? wk.chunk_cnt[kf] : 0;
    FF Q{0.f, 0.f};
    int64_t A = 0;
    if (seqs) {   // the sequences [s0, s1)
        for (int64_t base = s0 + 32 * warp; base < s1; base += kGrpoReduceThreads) {   // warp-uniform
            const int64_t s = base + lane;
            int64_t j0 = 0, j1 = -1;
            if (s < s1) {
                const bool first = base == s0 + 32 * warp;
                const int64_t a = first ? a_first : grpo_cu(p, s), e = first ? e_first : grpo_cu(p, s + 1);
                if (e > a) {
                    j0 = s + a / kGrpoChunk;
                    j1 = s + (e - 1) / kGrpoChunk;
                }
            }
            const bool is_long = j1 - j0 + 1 > kGrpoLongPieces;
            FF sum{0.f, 0.f};
            int64_t cnt = 0;
            if (!is_long) {   // up to 8 pieces per round, all loaded before they are added in order
                for (int64_t j = j0; j <= j1; j += 8) {
                    FF v[8];
                    int64_t c[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        v[u] = j + u <= j1 ? wk.piece[j + u] : FF{0.f, 0.f};
                        c[u] = j + u <= j1 ? wk.piece_cnt[j + u] : 0;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (j + u <= j1) {
                            sum = ff_add(sum, v[u]);
                            cnt += c[u];
                        }
                    }
                }
            }
            // the warp's long sequences, one at a time in lane order
            for (uint32_t m = __ballot_sync(0xffffffffu, is_long); m != 0; m &= m - 1) {
                const int src = __ffs(m) - 1;
                const int64_t k0 = __shfl_sync(0xffffffffu, j0, src), kl = __shfl_sync(0xffffffffu, j1, src);
                FF ws{0.f, 0.f};
                int64_t wc = 0;
                for (int64_t j = k0 + lane; j <= kl; j += 32) {
                    ws = ff_add(ws, wk.piece[j]);
                    wc += wk.piece_cnt[j];
                }
                ws = ff_warp_sum(ws);
                wc = warp_sum_i64(wc);
                const FF w0{__shfl_sync(0xffffffffu, ws.hi, 0), __shfl_sync(0xffffffffu, ws.lo, 0)};
                wc = __shfl_sync(0xffffffffu, wc, 0);
                if (lane == src) {
                    sum = w0;
                    cnt = wc;
                }
            }
            if (s < s1) {
                wk.seg_inv[s] = cnt > 0 ? __frcp_rn((float)cnt) : 0.f;
                if (cnt > 0) {
                    ++A;
                    if (p.mode == 1) Q = ff_add(Q, ff_div_count(sum, cnt));
                }
            }
        }
    }
    FF T = t_first;
    int64_t C = c_first;
    for (int64_t k = kf + kGrpoReduceThreads; k < k1; k += kGrpoReduceThreads) {
        T = ff_add(T, wk.chunk_sum[k]);
        C += wk.chunk_cnt[k];
    }
    T = cta_fold<kW>(T, C, sh_v, sh_c);
    if (seqs) Q = cta_fold<kW>(Q, A, sh_v, sh_c);
    if (G == 1) {
        if (threadIdx.x == 0) {
            wk.part_t[0] = T;
            wk.part_q[0] = Q;
            wk.part_c[0] = C;
            wk.part_a[0] = A;
        }
    } else {
        if (threadIdx.x == 0) {
            wk.part_t[b] = T;
            wk.part_q[b] = Q;
            wk.part_c[b] = C;
            wk.part_a[b] = A;
            __threadfence();
            last = atomicAdd(wk.ticket, 1u) == (unsigned)(G - 1);
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
    }
    // the last CTA: thread i takes partials i, i + 256, ... in order; the CTA
    // fold combines them (a fixed butterfly per warp, then warp order)
    FF t{0.f, 0.f}, q{0.f, 0.f};
    int64_t c = 0, a = 0;
    for (int i = threadIdx.x; i < G; i += kGrpoReduceThreads) {
        const float2 tv = __ldcg(reinterpret_cast<const float2*>(wk.part_t) + i);
        const float2 qv = __ldcg(reinterpret_cast<const float2*>(wk.part_q) + i);
        t = ff_add(t, FF{tv.x, tv.y});
        q = ff_add(q, FF{qv.x, qv.y});
        c += __ldcg(reinterpret_cast<const long long*>(wk.part_c) + i);
        a += __ldcg(reinterpret_cast<const long long*>(wk.part_a) + i);
    }
    t = cta_fold<kW>(t, c, sh_v, sh_c);
    q = cta_fold<kW>(q, a, sh_v, sh_c);
    if (threadIdx.x == 0) {
        const double tt = ff_value(t), cnt = (double)c;
        double qq = ff_value(q), aa = (double)a;
        if (!seqs) {   // the whole batch is one sequence (or token mean)
            aa = c > 0 ? 1.0 : 0.0;
            qq = c > 0 ? tt / cnt : 0.0;
        }
        double den = (p.mode == 0) ? cnt : aa;
        if (p.normalizer > 0.f) den = (double)p.normalizer;
        const double num = (p.mode == 1) ? qq : tt;
        p.loss[0] = den > 0 ? __double2float_rn(num / den) : 0.f;
        wk.den[0] = den;
        wk.den[1] = cnt;
        double w = 0.0;
        if (den > 0) w = (p.mode == 1 && p.cu == nullptr) ? (c > 0 ? 1.0 / (den * cnt) : 0.0) : 1.0 / den;
        wk.wt[0] = __double2float_rn(w);
        if (G > 1) *wk.ticket = 0u;
    }
}

// Each token's gradient times its weight: 1 / den, or for the sequence mean
// of token means with sequences 1 / (den n_s), n_s the sequence's active
// tokens (formed in FP32 as the product of the correctly rounded 1 / den and
// 1 / n_s, the latter kept per sequence by the fold).  Each warp takes a contiguous range of chunks (as in pass 1):
// the range's first sequence was recorded by pass 1, later chunks resume at
// the last sequence seen.
template <bool kVec>
__global__ void __launch_bounds__(kGrpoPassThreads, 5) k_grpo_scale(GrpoArgs p, GrpoWork wk) {
    const int lane = threadIdx.x & 31;
    const int64_t nchunks = grpo_chunks(p.n);
    griddep_wait();
    const double den = wk.den[0];
    const bool zero = !(den > 0);   // no active token: every gradient is 0 already (rewritten,
                                    // so that the lines kept in L2 by pass 1 are released)
    const float wu = zero ? 0.f : wk.wt[0];
    const uint64_t pol = l2_evict_first();
    const bool per_seq = !zero && p.mode == 1 && p.cu != nullptr;
    const float denf = (float)den;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t w_end = (gw + 1) * nchunks / nwarps;
    int64_t w = gw * nchunks / nwarps;
    int64_t s_resume = per_seq && w < w_end ? wk.chunk_first[w] : 0;
    const float inv_den = zero ? 0.f : __frcp_rn(denf);
    for (; w < w_end; ++w) {
        const int64_t c0 = w * kGrpoChunk;
        const int nv = (int)(p.n - c0 < kGrpoChunk ? p.n - c0 : kGrpoChunk);
        float g[kGrpoLaneTokens];
        grpo_ld8<kVec, true>(p.grad + c0, lane, nv, g, pol);
        if (per_seq) {
            const GrpoRuns runs = grpo_runs_at(p, s_resume, c0, lane, wk.seg_inv);
            int64_t s_last = runs.s;
            // each run's tokens times its weight; tokens in no sequence hold 0 already
            grpo_runs<true>(p, runs, c0, nv, lane, wk.seg_inv, [&](int64_t s, int ua, int ub, float inv_cnt) {
                s_last = s;
                const float ws = __fmul_rn(inv_den, inv_cnt);
                const uint32_t in = (ua == 0 && ub == nv) ? 0xffu : grpo_in8(lane, ua, ub);
#pragma unroll
                for (int q = 0; q < kGrpoLaneTokens; ++q)
                    if ((in >> q) & 1u) g[q] = __fmul_rn(g[q], ws);
            });
            s_resume = s_last;
        } else {
#pragma unroll
            for (int q = 0; q < kGrpoLaneTokens; ++q) g[q] = __fmul_rn(g[q], wu);
        }
        grpo_st8<kVec>(p.grad + c0, lane, nv, g, pol);
    }
}

}  // namespace flp
