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
// Every normaliser weight depends on the mask and the sequence layout only,
// so the counts come first and the token pass writes final gradients:
//   1. k_grpo_count (when there is a mask and the weight is not the
//      caller's): CTA b takes tokens [b R, (b + 1) R) in rounds of 32768,
//      counts the active tokens of each 16-token mask word, scans them in
//      token order and writes, with sequences, each word's prefix within the
//      range, and the range's total.  Integer counts: exact in any order.
//   2. k_grpo_fix: the ranges' exclusive prefix, a word's prefix and the
//      bits of the word below x give P(x), the active tokens before x, for
//      every sequence start x = cu_seqlens[s]: hence each sequence's count
//      n_s = P(cu[s + 1]) - P(cu[s]), per CTA the number of sequences with an
//      active token, and the active tokens D inside the sequences; it also
//      zeroes the ticket of pass 3's fold.  Pass 3's warps form the
//      normaliser and the weight from these.
//   3. k_grpo_pass: the batch is cut into fixed chunks of 256 tokens (one
//      warp each), independent of the sequence layout; each warp takes a
//      contiguous range of chunks.  It loads a chunk (8 tokens per lane in
//      two groups of 4, 16-byte accesses when the arrays allow) and finds
//      the sequences that cross it (for its first chunk a 32-ary search over
//      cu_seqlens, later resuming at the last sequence seen), overlapped with
//      the loads.  Each token's gradient is written once, with its weight
//      (1 / den, or 1 / (den n_s) for the sequence mean of token means);
//      each run (sequence s within the chunk) adds its loss sum (or, for the
//      sequence mean of means, that sum over n_s) to the warp's total.  The
//      CTA folds its warps in order; the CTA that finishes last (an atomic
//      ticket) folds the CTAs' sums in order into the loss.
// The grid of pass 3 and so every fold's shape are fixed by the problem's
// shape.  Within a 256-token chunk the sums are plain FP32 (each lane's 8
// tokens in order, then the xor butterfly: an error of at most about 12 u
// times the chunk's sum of |l|); from the chunk level up they are two-float
// (hi + lo) compensated sums in FP32 (Knuth's TwoSum per addition; the pair
// carries about 44 significant bits), so the error does not grow with the
// batch: the FP64 unit of this GPU is far too slow to accumulate per token.
// No fold's order depends on timing.
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
    uint64_t tag;               // the layout's tag (n, sequences, mode, normaliser, mask, cu_seqlens)
    int check_tag;              // pass 3: the counts come from an earlier call; check their tag
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

// Pass 3's grid for a large batch: one wave of 4 CTAs per SM on a 152-SM
// GB300, a constant so that the fold's shape depends on the problem only.
constexpr int kGrpoPassCtas = 608;
// The count: 256 threads, 8 mask words of 16 tokens per thread per round,
// at most 1024 ranges (the fix kernel scans them in one CTA of 1024 threads).
constexpr int kGrpoCountThreads = 256;
constexpr int kGrpoCountWords = 8;
constexpr int64_t kGrpoCountRound = 16 * kGrpoCountWords * kGrpoCountThreads;   // 32768 tokens
constexpr int kGrpoCountMaxCtas = 1024;
// The sequences' counts: one sequence per thread and step, at most 1024
// CTAs of 256 threads.
constexpr int kGrpoFixThreads = 256;
constexpr int kGrpoFixMaxCtas = 1024;

// e^x as 2^(x log2 e), the power of two from the special-function unit
// (ex2.approx, flushing subnormal results to 0): within a few ulp for
// |x| <~ 1, the error growing by about |x| 2^-24 from rounding x log2 e.
__device__ __forceinline__ float grpo_exp(float x) { return ex2_ftz(__fmul_rn(x, 1.4426950408889634f)); }

struct GrpoWork {
    int64_t* dcnt;        // [1]: active tokens inside the sequences (or in the batch)
    unsigned* ticket;     // [1]: CTAs of pass 3 that are done (zeroed by the fix kernel, counted by
                          //      pass 3, zeroed again by its last CTA)
    uint64_t* tag;        // [1]: the tag of the layout the counts were taken for
    FF* part_t;           // [kGrpoPassCtas]: per CTA of pass 3, its loss sum
    FF* part_q;           //   its sum of sequence means' pieces
    int64_t* a_part;      // [kGrpoFixMaxCtas]: per CTA of the fix kernel, its sequences with an active token
    int64_t* range_cnt;   // [kGrpoCountMaxCtas]: active tokens of each count range
    uint32_t* word_pre;   // [ceil(n / 16)] with sequences: active tokens of a word's range before the word
    float2* seg_cnt;      // [nseq]: active tokens of each sequence n_s and 1 / n_s (0 for none), FP32
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
    float2 aux;    // lane j: aux[s + j] when an aux array is given (s + j < nseq), else 0
};

__device__ __forceinline__ GrpoRuns grpo_runs_at(const GrpoArgs& p, int64_t s, int64_t c0, int lane,
                                                 const float2* aux) {
    GrpoRuns r{s < 0 ? 0 : s, (int)kGrpoChunk, make_float2(0.f, 0.f)};
    const int64_t idx = r.s + lane;
    if (idx <= p.nseq) {
        const int64_t d = grpo_cu(p, idx) - c0;
        r.bnd = d < 0 ? 0 : (d > kGrpoChunk ? (int)kGrpoChunk : (int)d);
    }
    if (aux && idx < p.nseq) r.aux = aux[idx];
    return r;
}
__device__ __forceinline__ GrpoRuns grpo_runs_begin(const GrpoArgs& p, int64_t c0, int lane) {
    if (p.cu == nullptr) return GrpoRuns{0, 0, make_float2(0.f, 0.f)};
    return grpo_runs_at(p, grpo_find(p, c0, lane), c0, lane, nullptr);
}

__device__ __forceinline__ float2 shfl_f2(float2 v, int src) {
    return make_float2(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src));
}

// Calls f(s, ua, ub, aux_s) for each sequence s whose tokens meet the chunk
// of nv tokens from c0, in sequence order, with [ua, ub) the chunk-local
// indices of its tokens there (never empty).  Warp-uniform; boundaries are
// fetched 32 at a time.  kAux: pass the aux value (else 0, no shuffle).
template <bool kAux, class F>
__device__ __forceinline__ void grpo_runs(const GrpoArgs& p, GrpoRuns r, int64_t c0, int nv, int lane,
                                          const float2* aux, F&& f) {
    if (p.cu == nullptr) {
        f((int64_t)0, 0, nv, make_float2(0.f, 0.f));   // one sequence: the whole batch
        return;
    }
    if (r.s < p.nseq) {   // the common case: the chunk lies inside sequence r.s
        const int a0 = __shfl_sync(0xffffffffu, r.bnd, 0), b0 = __shfl_sync(0xffffffffu, r.bnd, 1);
        if (a0 == 0 && b0 >= nv) {
            f(r.s, 0, nv, kAux ? shfl_f2(r.aux, 0) : make_float2(0.f, 0.f));
            return;
        }
    }
    while (r.s < p.nseq) {
        for (int j = 0; j < 31; ++j) {
            const int a = __shfl_sync(0xffffffffu, r.bnd, j);
            if (r.s + j >= p.nseq || a >= nv) return;
            const int b = min(__shfl_sync(0xffffffffu, r.bnd, j + 1), nv);
            const float2 x = kAux ? shfl_f2(r.aux, j) : make_float2(0.f, 0.f);
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

// Bits of the 16 mask bytes from token u (those at or past `end` left 0):
// bit i set when byte u + i is nonzero.  kVec: one 16-byte load (the mask
// 16-byte aligned, u a multiple of 16); it keeps the default L2 policy, so
// that pass 3's read of the same bytes may still find them there.
template <bool kVec>
__device__ __forceinline__ uint32_t grpo_mask_bits16(const uint8_t* mask, int64_t u, int64_t end) {
    if (kVec && u + 16 <= end) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(mask + u));
        const uint32_t x[4] = {w.x, w.y, w.z, w.w};
        uint32_t b = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) b |= (((__vcmpne4(x[i], 0u) & 0x01010101u) * 0x01020408u) >> 24) << (4 * i);
        return b;
    }
    uint32_t b = 0;
    for (int i = 0; i < 16; ++i)
        if (u + i < end && __ldg(mask + u + i) != 0) b |= 1u << i;
    return b;
}

// Pass 1: the active tokens of each range of `range` tokens (a multiple of
// 16) and, when there are sequences, of each 16-token word's range before
// the word.  A round's word counts go through shared memory so that thread
// t scans words [8 t, 8 t + 8) after the CTA's exclusive scan of the
// threads' sums: the prefix runs in token order.
template <bool kVec>
__global__ void __launch_bounds__(kGrpoCountThreads) k_grpo_count(GrpoArgs p, GrpoWork wk, int64_t range) {
    constexpr int kWords = kGrpoCountWords * kGrpoCountThreads;
    __shared__ uint8_t sh_cnt[kWords];
    __shared__ uint32_t sh_pre[kWords];
    __shared__ uint32_t sh_wsum[kGrpoCountThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t t0 = (int64_t)blockIdx.x * range;
    const int64_t t1 = t0 + range < p.n ? t0 + range : p.n;
    griddep_launch_dependents();
    int64_t base = 0;   // active tokens in [t0, r0)
    for (int64_t r0 = t0; r0 < t1; r0 += kGrpoCountRound) {
        const int64_t r1 = r0 + kGrpoCountRound < t1 ? r0 + kGrpoCountRound : t1;
        uint32_t bits[kGrpoCountWords];
        if (kVec) {   // every whole word's load first (predicated, no branch), then the bits
            uint4 wv[kGrpoCountWords];
#pragma unroll
            for (int k = 0; k < kGrpoCountWords; ++k) {
                const int64_t u = r0 + 16 * (int64_t)(k * kGrpoCountThreads + tid);
                wv[k] = u + 16 <= r1 ? __ldg(reinterpret_cast<const uint4*>(p.mask + u)) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < kGrpoCountWords; ++k) {
                const int64_t u = r0 + 16 * (int64_t)(k * kGrpoCountThreads + tid);
                const uint32_t x[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
                uint32_t b = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) b |= (((__vcmpne4(x[i], 0u) & 0x01010101u) * 0x01020408u) >> 24) << (4 * i);
                bits[k] = (u < r1 && u + 16 > r1) ? grpo_mask_bits16<false>(p.mask, u, r1) : b;   // the ragged end
            }
        } else {
#pragma unroll
            for (int k = 0; k < kGrpoCountWords; ++k) {
                const int64_t u = r0 + 16 * (int64_t)(k * kGrpoCountThreads + tid);
                bits[k] = u < r1 ? grpo_mask_bits16<false>(p.mask, u, r1) : 0u;
            }
        }
#pragma unroll
        for (int k = 0; k < kGrpoCountWords; ++k) sh_cnt[k * kGrpoCountThreads + tid] = (uint8_t)__popc(bits[k]);
        __syncthreads();
        uint32_t c[kGrpoCountWords], sum = 0;
#pragma unroll
        for (int i = 0; i < kGrpoCountWords; ++i) {
            c[i] = sh_cnt[kGrpoCountWords * tid + i];
            sum += c[i];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) sh_wsum[warp] = incl;
        __syncthreads();
        uint32_t run = incl - sum, total = 0;
#pragma unroll
        for (int w = 0; w < kGrpoCountThreads / 32; ++w) {
            const uint32_t x = sh_wsum[w];
            run += w < warp ? x : 0u;
            total += x;
        }
        if (p.cu != nullptr) {   // through shared memory, so that the stores are coalesced
#pragma unroll
            for (int i = 0; i < kGrpoCountWords; ++i) {
                sh_pre[kGrpoCountWords * tid + i] = (uint32_t)base + run;
                run += c[i];
            }
            __syncthreads();
            const int64_t wn = ((r1 + 15) >> 4) - (r0 >> 4);   // words of the round
#pragma unroll
            for (int k = 0; k < kGrpoCountWords; ++k) {
                const int j = k * kGrpoCountThreads + tid;
                if (j < wn) wk.word_pre[(r0 >> 4) + j] = sh_pre[j];
            }
        }
        base += total;
        __syncthreads();   // the next round rewrites the shared arrays
    }
    if (tid == 0) wk.range_cnt[blockIdx.x] = base;
}

// Pass 2: thread t of CTA b takes sequence s = 256 b + t (then s + 256 G,
// ...).  Its two bounds are loaded first; while they are in flight the CTA
// scans the ranges' counts (with a mask; else every token is active); then
// the word prefix and the mask word at each bound are loaded together, and
// P(x) = the ranges before x + the word's prefix in its range + the word's
// active tokens below x.  n_s = P(cu[s + 1]) - P(cu[s]) and its correctly
// rounded reciprocal are written for the sequence mean of token means; each CTA writes its number of sequences
// with an active token (not needed for the token mean).  CTA 0 writes the
// active tokens D inside the sequences (or in the batch), zeroes pass 3's
// ticket and writes the loss when there are no tokens.
template <bool kVec>
__global__ void __launch_bounds__(kGrpoFixThreads) k_grpo_fix(GrpoArgs p, GrpoWork wk, int64_t range, int nranges) {
    constexpr int kW = kGrpoFixThreads / 32;
    constexpr int kPer = kGrpoCountMaxCtas / kGrpoFixThreads;     // ranges per thread in the scan
    __shared__ int64_t sh_pre[kGrpoCountMaxCtas];
    __shared__ int64_t sh_w[kW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_launch_dependents();
    griddep_wait();
    const bool counted = p.mask != nullptr && nranges > 0;
    const bool per_seq = p.cu != nullptr && p.n > 0 && p.mode != 0;   // with no tokens cu_seqlens is not read
    const int64_t step = (int64_t)gridDim.x * kGrpoFixThreads;
    int64_t s = (int64_t)blockIdx.x * kGrpoFixThreads + tid;
    int64_t xa = p.n, xb = p.n;
    if (per_seq && s < p.nseq) {
        xa = grpo_cu(p, s);
        xb = grpo_cu(p, s + 1);
    }
    int64_t total = p.n;
    if (counted) {   // thread t scans ranges [kPer t, kPer t + kPer)
        int64_t v[kPer], sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int r = kPer * tid + i;
            v[i] = r < nranges ? __ldcg(reinterpret_cast<const long long*>(wk.range_cnt) + r) : 0;
            sum += v[i];
        }
        int64_t incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) sh_w[warp] = incl;
        __syncthreads();
        int64_t run = incl - sum;
        total = 0;
        for (int w = 0; w < kW; ++w) {
            const int64_t x = sh_w[w];
            run += w < warp ? x : 0;
            total += x;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            sh_pre[kPer * tid + i] = run;
            run += v[i];
        }
        __syncthreads();
    }
    // the two loads of P(x) (none without a mask or at the end of the batch)
    auto loads_at = [&](int64_t x, uint32_t& wpre, uint32_t& wbits) {
        wpre = 0;
        wbits = 0;
        if (counted && x < p.n) {
            wpre = __ldcg(wk.word_pre + (x >> 4));
            wbits = grpo_mask_bits16<kVec>(p.mask, x & ~(int64_t)15, p.n);
        }
    };
    auto active_before = [&](int64_t x, uint32_t wpre, uint32_t wbits) -> int64_t {
        if (!counted) return x;
        if (x >= p.n) return total;
        return sh_pre[x / range] + (int64_t)wpre + __popc(wbits & ((1u << (x & 15)) - 1u));
    };
    int64_t A = 0;
    while (per_seq && s < p.nseq) {
        uint32_t pa, ba, pb, bb;
        loads_at(xa, pa, ba);
        loads_at(xb, pb, bb);
        int64_t c = active_before(xb, pb, bb) - active_before(xa, pa, ba);
        c = c < 0 ? 0 : c;
        if (p.mode == 1) {
            const float cf = (float)c;
            wk.seg_cnt[s] = make_float2(cf, c > 0 ? __frcp_rn(cf) : 0.f);
        }
        A += c > 0 ? 1 : 0;
        s += step;
        if (s < p.nseq) {
            xa = grpo_cu(p, s);
            xb = grpo_cu(p, s + 1);
        }
    }
    A = warp_sum_i64(A);
    __syncthreads();   // sh_w is reused
    if (lane == 0) sh_w[warp] = A;
    __syncthreads();
    if (tid == 0) {
        A = 0;
        for (int w = 0; w < kW; ++w) A += sh_w[w];
        wk.a_part[blockIdx.x] = A;
        if (blockIdx.x == 0) {
            int64_t D = total;
            if (p.cu != nullptr && p.n > 0) {
                const int64_t x0 = grpo_cu(p, 0), x1 = grpo_cu(p, p.nseq);
                uint32_t pa, ba, pb, bb;
                loads_at(x0, pa, ba);
                loads_at(x1, pb, bb);
                D = active_before(x1, pb, bb) - active_before(x0, pa, ba);
                D = D < 0 ? 0 : D;
            }
            *wk.dcnt = D;
            *wk.ticket = 0u;
            *wk.tag = p.tag;
            if (p.n == 0 && p.loss != nullptr) p.loss[0] = 0.f;
        }
    }
}

// The normaliser and the uniform weight from the active tokens D and the
// number A of sequences with an active token.
struct GrpoNorm {
    double den, cnt;
    float wt;
};
__device__ __forceinline__ GrpoNorm grpo_norm(const GrpoArgs& p, int64_t A, int64_t D) {
    const bool seqs = p.cu != nullptr && p.mode != 0 && p.n > 0;
    const double cnt = (double)D;
    const double aa = seqs ? (double)A : (D > 0 ? 1.0 : 0.0);
    double den = (p.mode == 0) ? cnt : aa;
    if (p.normalizer > 0.f) den = (double)p.normalizer;
    double w = 0.0;
    if (den > 0) w = (p.mode == 1 && p.cu == nullptr) ? (D > 0 ? 1.0 / (den * cnt) : 0.0) : 1.0 / den;
    return {den, cnt, __double2float_rn(w)};
}
// The same on every lane of a warp: the fix kernel's A partials summed.
__device__ __forceinline__ GrpoNorm grpo_norm_warp(const GrpoArgs& p, const GrpoWork& wk, int nfix, int lane) {
    int64_t A = 0;
    for (int i = lane; i < nfix; i += 32) A += __ldcg(reinterpret_cast<const long long*>(wk.a_part) + i);
    A = warp_sum_i64(A);
    return grpo_norm(p, A, __ldcg(reinterpret_cast<const long long*>(wk.dcnt)));
}

// A sequence's piece s over its active count c as two floats, from the
// correctly rounded reciprocal inv = 1 / c: q = s inv, and the residual
// s - q c (one rounding, by the fused multiply-add) times inv as the low
// part, so that q + lo carries s / c to about 2^-46 relative.
__device__ __forceinline__ FF ff_div_countf(float s, float c, float inv) {
    const float q = __fmul_rn(s, inv);
    const float r = __fmaf_rn(-q, c, s);
    return {q, __fmul_rn(r, inv)};
}

// Folds v over the CTA: the fixed butterfly in each warp, then warp order
// (thread 0 gets the result; every thread must call it).
template <int kWarps>
__device__ __forceinline__ FF cta_fold(FF v, FF* sh_v) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = ff_warp_sum(v);
    __syncthreads();   // the shared slots may still be read by a previous fold
    if (lane == 0) sh_v[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        v = FF{0.f, 0.f};
        for (int w = 0; w < kWarps; ++w) v = ff_add(v, sh_v[w]);
    }
    return v;
}

// Pass 3 (see the top of this file).  kSeq: the sequence mean of token
// means with sequences, i.e. a weight per sequence.  The weight is the
// caller's (p.prescale > 0: the fix kernel is waited for only before the
// ticket) or the fix kernel's (waited for first).
template <bool kVec, bool kSeq>
__global__ void __launch_bounds__(kGrpoPassThreads, 4) k_grpo_pass(GrpoArgs p, GrpoWork wk, int nfix) {
    constexpr int kW = kGrpoPassThreads / 32;
    __shared__ FF sh_t[kW], sh_q[kW];
    __shared__ bool last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nchunks = grpo_chunks(p.n);
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const float clo = 1.f - p.eps_lo, chi = 1.f + p.eps_hi;
    griddep_launch_dependents();
    const uint64_t pol = l2_evict_first();
    const bool known = p.prescale > 0.f;
    float wu = p.prescale, inv_den = 0.f;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t w_end = (gw + 1) * nchunks / nwarps;
    // counts from an earlier call taken for another layout: every gradient
    // and the loss become NaN
    bool stale = false;
    if (!known) {   // the counts and the weight
        griddep_wait();
        const GrpoNorm nm = grpo_norm_warp(p, wk, nfix, lane);
        stale = p.check_tag && __ldcg(reinterpret_cast<const unsigned long long*>(wk.tag)) != p.tag;
        wu = stale ? __int_as_float(0x7fc00000) : nm.wt;
        inv_den = stale ? __int_as_float(0x7fc00000) : (nm.den > 0 ? __frcp_rn((float)nm.den) : 0.f);
    }
    FF T{0.f, 0.f}, Q{0.f, 0.f};
    int64_t s_resume = -1;
    for (int64_t w = gw * nchunks / nwarps; w < w_end; ++w) {
        const int64_t c0 = w * kGrpoChunk;
        const int nv = (int)(p.n - c0 < kGrpoChunk ? p.n - c0 : kGrpoChunk);   // tokens in the chunk
        float lp[kGrpoLaneTokens], od[kGrpoLaneTokens], av[kGrpoLaneTokens], rf[kGrpoLaneTokens];
        grpo_ld8<kVec>(p.logp + c0, lane, nv, lp, pol);
        grpo_ld8<kVec>(p.old_logp + c0, lane, nv, od, pol);
        grpo_ld8<kVec>(p.adv + c0, lane, nv, av, pol);
        if (p.ref_logp) grpo_ld8<kVec>(p.ref_logp + c0, lane, nv, rf, pol);
        const uint32_t act = grpo_active8<kVec>(p.mask ? p.mask + c0 : nullptr, lane, nv, pol);
        // overlaps the loads above
        const GrpoRuns runs = (s_resume < 0 || p.cu == nullptr)
                                  ? (kSeq ? grpo_runs_at(p, grpo_find(p, c0, lane), c0, lane, wk.seg_cnt)
                                          : grpo_runs_begin(p, c0, lane))
                                  : grpo_runs_at(p, s_resume, c0, lane, kSeq ? wk.seg_cnt : nullptr);
        int64_t s_last = runs.s;
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
        uint32_t inseq = 0;
        grpo_runs<kSeq>(p, runs, c0, nv, lane, kSeq ? wk.seg_cnt : nullptr,
                        [&](int64_t s, int ua, int ub, float2 cnt_s) {
            s_last = s;
            // within the chunk, plain FP32: the lane's tokens in order, then the
            // xor butterfly (every lane holds the result)
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
            if (kSeq && p.cu) {
                // the run's tokens times 1 / (den n_s): the product of the correctly
                // rounded 1 / den and 1 / n_s
                const float ws = __fmul_rn(inv_den, cnt_s.y);
                if (in == 0xffu) {
#pragma unroll
                    for (int q = 0; q < kGrpoLaneTokens; ++q) dl[q] = __fmul_rn(dl[q], ws);
                } else {
#pragma unroll
                    for (int q = 0; q < kGrpoLaneTokens; ++q)
                        if ((in >> q) & 1u) dl[q] = __fmul_rn(dl[q], ws);
                }
                if (cnt_s.x > 0.f) Q = ff_add(Q, ff_div_countf(rs, cnt_s.x, cnt_s.y));
            }
            tot = ff_add(tot, rs);
        });
        if (p.cu && inseq != 0xffu) {   // tokens outside every sequence
#pragma unroll
            for (int q = 0; q < kGrpoLaneTokens; ++q) {
                const bool in = (inseq >> q) & 1u;
                l[q] = in ? l[q] : 0.f;
                dl[q] = in ? dl[q] : 0.f;
            }
        }
        if (!(kSeq && p.cu)) {   // one weight for every token
#pragma unroll
            for (int q = 0; q < kGrpoLaneTokens; ++q) dl[q] = __fmul_rn(dl[q], wu);
        }
        grpo_st8<kVec>(p.grad + c0, lane, nv, dl, pol);
        if (p.token_loss) grpo_st8<kVec>(p.token_loss + c0, lane, nv, l, pol);
        T = ff_add(T, tot);
        s_resume = s_last;   // no later chunk meets an earlier sequence
    }
    if (known) griddep_wait();   // the ticket and the normaliser
    // the CTA's sums (every lane of a warp holds its warp's), warps in order
    if (lane == 0) {
        sh_t[warp] = T;
        sh_q[warp] = Q;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        FF t{0.f, 0.f}, q{0.f, 0.f};
        for (int i = 0; i < kW; ++i) {
            t = ff_add(t, sh_t[i]);
            q = ff_add(q, sh_q[i]);
        }
        wk.part_t[blockIdx.x] = t;
        wk.part_q[blockIdx.x] = q;
        __threadfence();
        last = atomicAdd(wk.ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    // the last CTA: thread i takes the CTAs i, i + 256, ... in order, then the
    // CTA fold (a fixed butterfly per warp, then warp order)
    FF t{0.f, 0.f}, q{0.f, 0.f};
    for (int i = threadIdx.x; i < (int)gridDim.x; i += kGrpoPassThreads) {
        const float2 tv = __ldcg(reinterpret_cast<const float2*>(wk.part_t) + i);
        const float2 qv = __ldcg(reinterpret_cast<const float2*>(wk.part_q) + i);
        t = ff_add(t, FF{tv.x, tv.y});
        q = ff_add(q, FF{qv.x, qv.y});
    }
    t = cta_fold<kW>(t, sh_t);
    q = cta_fold<kW>(q, sh_q);
    const GrpoNorm nm = warp == 0 ? grpo_norm_warp(p, wk, nfix, lane) : GrpoNorm{0.0, 0.0, 0.f};
    if (threadIdx.x == 0) {
        const double den = nm.den, cnt = nm.cnt;
        const double tt = ff_value(t);
        double num = tt;
        if (p.mode == 1) num = p.cu ? ff_value(q) : (cnt > 0 ? tt / cnt : 0.0);
        p.loss[0] = stale ? __int_as_float(0x7fc00000) : (den > 0 ? __double2float_rn(num / den) : 0.f);
        *wk.ticket = 0u;   // every CTA has counted: ready for a call that reuses the counts
    }
}

}  // namespace flp
