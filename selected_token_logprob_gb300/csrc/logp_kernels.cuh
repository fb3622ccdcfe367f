// Device code of the selected-token log-probability path for sm_103a.
//
// Forward (RL-Kernel issue #241 "TP-aware deterministic logprob", Background
// and PR 3 bullets): LSE_t = log sum_v exp(x[t, v]) with FP32 accumulation,
// logp_t = x[t, y_t] - LSE_t.  One CTA per row, one warp per vocabulary tile
// (16 tiles of width W = 8 * ceil(V / 128)): each lane keeps an online
// (max, sumexp) pair over its fixed share of the tile, the warp merges the 32
// pairs with a fixed xor butterfly, and a half-warp merges the 16 tile
// partials with a fixed pairwise tree in tile-index order (RL-Kernel PR #314,
// tensor-parallel section: fixed tiles, one fixed merge order).  Nothing in
// this order depends on N, on the row's position or on the grid, so every
// row's bits are batch-invariant, and a vocab shard that reduces its own tiles
// with the same functions reproduces the same partials bit for bit.
//
// Backward (RL-Kernel PR #495 "zero-workspace fused backward", Summary item
// 2): dlogits = g * (onehot - exp(x - LSE)) from the saved LSE, one read and
// one write per logit, elementwise.
//
// All index arithmetic is 64-bit.  No kernel waits on another CTA.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace flp {

constexpr int kTiles = 16;                  // vocabulary tiles per row (K)
constexpr int kWarp = 32;
constexpr int kFwdThreads = kTiles * kWarp; // one warp per tile
constexpr int kGroup = 4;                   // 16-byte vectors per lane per online step
constexpr int kBwdThreads = 256;
constexpr int kBwdVecPerThread = 4;
constexpr int64_t kBwdSegCols = (int64_t)kBwdThreads * kBwdVecPerThread * 8;

// Mathematical constants: ln 2 to double precision, its binary32 head and
// tail (so that head + tail = ln 2 to about 2^-48 relative), and log2(e)
// rounded to binary32.
constexpr double kLn2 = 0.6931471805599453094172321214581766;
constexpr float kLn2Hi = (float)kLn2;
constexpr float kLn2Lo = (float)(kLn2 - (double)kLn2Hi);
constexpr float kLog2e = (float)(1.0 / kLn2);

struct MS {
    float m;  // running maximum (always the value of an input element, or -inf)
    float s;  // sum of exp(x - m) over the elements seen
};

// ---------------------------------------------------------------- loads

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}

__device__ __forceinline__ void st_cs_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// A BF16 value is the top half of a binary32: widening is a shift.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf_scalar(const uint16_t* p) {
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p)) << 16);
}

// Two binary32 -> packed BF16 pair, round to nearest even (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^a on the special-function unit; results below 2^-126 flush to zero
// (they are below 2^-126 of the running maximum's own term, which is 1).
__device__ __forceinline__ float ex2_ftz(float a) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// 2^a on the special-function unit, keeping subnormal results.
__device__ __forceinline__ float ex2_full(float a) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// Eight consecutive columns [col, col + 8) of a tile; columns >= width read
// as -inf (padded columns are masked, PR #314 ReductionSpec).  The vector
// path needs a 16-byte aligned tile base; both paths yield the same floats.
template <bool kVec>
__device__ __forceinline__ void load8(const uint16_t* __restrict__ tile, int64_t col,
                                      int64_t width, float (&f)[8]) {
    if (kVec && col + 8 <= width) {
        const uint4 q = ld_nc_v4(tile + col);
        f[0] = bf_lo(q.x); f[1] = bf_hi(q.x);
        f[2] = bf_lo(q.y); f[3] = bf_hi(q.y);
        f[4] = bf_lo(q.z); f[5] = bf_hi(q.z);
        f[6] = bf_lo(q.w); f[7] = bf_hi(q.w);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            f[j] = (col + j < width) ? bf_scalar(tile + col + j) : -INFINITY;
    }
}

// ---------------------------------------------------------------- forward reduction

// Online (max, sumexp) of one lane over its share of a tile of `width`
// columns: 16-byte vector j of the tile belongs to lane j mod 32, and the
// lane visits its vectors in increasing j, kGroup at a time.  Per group:
// the group maximum gm = max(m, group elements); each vector's eight terms
// exp(x - gm) are summed as a fixed pairwise tree, the kGroup vector sums as
// another; then s = s * exp(m - gm) + group sum (one fused multiply-add).
// x - gm is exact (both are BF16 values), so exp(x - gm) is 2^((x - gm)
// log2 e) with only the product rounded.
template <bool kVec>
__device__ __forceinline__ MS tile_scan(const uint16_t* __restrict__ tile, int64_t width,
                                        int lane) {
    const int64_t nvec = (width + 7) >> 3;
    float m = -INFINITY, s = 0.f;
    for (int64_t v0 = 0; v0 < nvec; v0 += (int64_t)kWarp * kGroup) {
        float f[kGroup][8];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int64_t j = v0 + lane + (int64_t)kWarp * u;
            if (j < nvec) {
                load8<kVec>(tile, j * 8, width, f[u]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[u][e] = -INFINITY;
            }
        }
        float gm = m;
#pragma unroll
        for (int u = 0; u < kGroup; ++u)
#pragma unroll
            for (int e = 0; e < 8; ++e) gm = fmaxf(gm, f[u][e]);
        if (gm == -INFINITY) continue;  // nothing finite seen yet: (m, s) stays (-inf, 0)
        float vs[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            if (v0 + lane + (int64_t)kWarp * u < nvec) {
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) p[e] = ex2_ftz(__fmul_rn(__fsub_rn(f[u][e], gm), kLog2e));
                vs[u] = __fadd_rn(__fadd_rn(__fadd_rn(p[0], p[1]), __fadd_rn(p[2], p[3])),
                                  __fadd_rn(__fadd_rn(p[4], p[5]), __fadd_rn(p[6], p[7])));
            } else {
                vs[u] = 0.f;
            }
        }
        static_assert(kGroup == 4, "group tree below is written for four vectors");
        const float gs = __fadd_rn(__fadd_rn(vs[0], vs[1]), __fadd_rn(vs[2], vs[3]));
        const float r = (m == gm) ? 1.f : ex2_ftz(__fmul_rn(__fsub_rn(m, gm), kLog2e));
        s = __fmaf_rn(s, r, gs);
        m = gm;
    }
    return MS{m, s};
}

// Merge of two (max, sumexp) pairs: the pair holding the larger max keeps its
// sum, the other is scaled by exp(m_small - M).  Symmetric in its arguments
// (IEEE addition commutes), so both lanes of a butterfly get the same bits.
__device__ __forceinline__ MS ms_merge(MS a, MS b) {
    const bool a_big = a.m >= b.m;
    const float M = a_big ? a.m : b.m;
    const float m_small = a_big ? b.m : a.m;
    const float s_big = a_big ? a.s : b.s;
    const float s_small = a_big ? b.s : a.s;
    float r;
    if (m_small == -INFINITY) r = 0.f;
    else if (m_small == M) r = 1.f;
    else r = ex2_ftz(__fmul_rn(__fsub_rn(m_small, M), kLog2e));
    return MS{M, __fmaf_rn(s_small, r, s_big)};
}

// Fixed xor butterfly over the 32 lanes of a warp (offsets 16, 8, 4, 2, 1);
// every lane ends with the same pair.
__device__ __forceinline__ MS warp_merge(MS p) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        MS o;
        o.m = __shfl_xor_sync(0xffffffffu, p.m, off);
        o.s = __shfl_xor_sync(0xffffffffu, p.s, off);
        p = ms_merge(p, o);
    }
    return p;
}

// Merge of the 16 tile partials of one row held by a 16-lane half warp
// (lane k of the half holds tile k; tiles k >= n_tiles hold the identity
// (-inf, 0)).  M = max m_k; S = sum_k s_k exp(m_k - M) summed as a fixed
// pairwise tree in tile-index order (issue #241 PR 3 merge formula).  The
// exponent argument m_k - M is exact; exp is the accurate library expf.
// All 32 lanes must call this together.  Returns (M, S) in every lane.
__device__ __forceinline__ MS tile_fold16(MS p) {
    float M = p.m;
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off, 16));
    float term = (p.m == -INFINITY) ? 0.f : __fmul_rn(p.s, expf(__fsub_rn(p.m, M)));
#pragma unroll
    for (int off = 1; off <= 8; off <<= 1) term = __fadd_rn(term, __shfl_xor_sync(0xffffffffu, term, off, 16));
    return MS{M, term};
}

// LSE = M + log S and logp = x_y - LSE, the log and both subtractions carried
// in double and each output rounded once to binary32 (the "downcast at final
// write" of issue #241 Goal).
__device__ __forceinline__ void finalize_row(MS f, bool active, float x_y, float* logp_out,
                                             float* lse_out) {
    const double l = (f.m == -INFINITY) ? -(double)INFINITY : (double)f.m + log((double)f.s);
    *lse_out = __double2float_rn(l);
    *logp_out = active ? __double2float_rn((double)x_y - l) : 0.f;
}

__device__ __forceinline__ bool row_active(int64_t y, int64_t v, int64_t ignore_index) {
    return y >= 0 && y < v && y != ignore_index;
}

// ---------------------------------------------------------------- kernels

// Forward: one CTA (16 warps) per row, warp k reduces tile k.
template <bool kVec>
__global__ void __launch_bounds__(kFwdThreads)
k_logp_fwd(const uint16_t* __restrict__ x, int64_t n, int64_t v, int64_t ld, int64_t W,
           const int64_t* __restrict__ y, int64_t ignore_index, float* __restrict__ logp,
           float* __restrict__ lse) {
    __shared__ float sh_m[kTiles], sh_s[kTiles];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
        const uint16_t* __restrict__ xr = x + t * ld;
        // the target and its logit are fetched early so their latency hides
        // behind the streaming
        bool act = false;
        float x_y = 0.f;
        if (threadIdx.x == 0) {
            const int64_t yt = __ldg(y + t);
            act = row_active(yt, v, ignore_index);
            if (act) x_y = bf_scalar(xr + yt);
        }
        const int64_t c0 = (int64_t)warp * W;
        const int64_t width = c0 >= v ? 0 : (v - c0 < W ? v - c0 : W);
        MS p = tile_scan<kVec>(xr + c0, width, lane);
        p = warp_merge(p);
        if (lane == 0) {
            sh_m[warp] = p.m;
            sh_s[warp] = p.s;
        }
        __syncthreads();
        if (warp == 0) {
            const int k = lane & 15;
            MS f = tile_fold16(MS{sh_m[k], sh_s[k]});
            if (lane == 0) finalize_row(f, act, x_y, logp + t, lse + t);
        }
        __syncthreads();
    }
}

// Shard partials: one CTA per row, warp w reduces the shard's local tile w
// (global tile tile0 + w) with the same tile_scan/warp_merge as the forward.
template <bool kVec>
__global__ void __launch_bounds__(kFwdThreads)
k_logp_partials(const uint16_t* __restrict__ xs, int64_t n, int64_t ld, int64_t real_width,
                int64_t W, int tile0, int64_t vocab_start, const int64_t* __restrict__ y,
                float* __restrict__ pm, float* __restrict__ ps, float* __restrict__ sel) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
        const uint16_t* __restrict__ xr = xs + t * ld;
        if (threadIdx.x == 0) {
            const int64_t yt = __ldg(y + t);
            if (yt >= vocab_start && yt < vocab_start + real_width)
                sel[t] = bf_scalar(xr + (yt - vocab_start));
        }
        const int64_t c0 = (int64_t)warp * W;
        const int64_t width = real_width - c0 < W ? real_width - c0 : W;
        MS p = tile_scan<kVec>(xr + c0, width, lane);
        p = warp_merge(p);
        if (lane == 0) {
            pm[t * kTiles + tile0 + warp] = p.m;
            ps[t * kTiles + tile0 + warp] = p.s;
        }
    }
}

// Merge of tile partials: one half warp per row, the same tile_fold16 and
// finalize_row as the forward.
__global__ void __launch_bounds__(256)
k_logp_merge(const float* __restrict__ pm, const float* __restrict__ ps,
             const float* __restrict__ sel, const int64_t* __restrict__ y,
             int64_t ignore_index, int64_t n, int64_t v, int n_tiles,
             float* __restrict__ logp, float* __restrict__ lse) {
    const int lane = threadIdx.x & 31, k = lane & 15;
    const int64_t warp_g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t pair = warp_g; 2 * pair < n; pair += n_warps) {
        const int64_t t = 2 * pair + (lane >> 4);
        const bool valid = t < n;
        MS p{-INFINITY, 0.f};
        if (valid && k < n_tiles) {
            p.m = __ldg(pm + t * kTiles + k);
            p.s = __ldg(ps + t * kTiles + k);
        }
        MS f = tile_fold16(p);
        if (valid && k == 0) {
            const int64_t yt = __ldg(y + t);
            const bool act = row_active(yt, v, ignore_index);
            const float x_y = act ? __ldg(sel + t) : 0.f;
            finalize_row(f, act, x_y, logp + t, lse + t);
        }
    }
}

// Backward: one CTA per (row, segment of kBwdSegCols columns).  Per active
// row: lse is split as lse_r + delta with lse_r on a 2^-16 grid, so that
// t = x - lse_r is exact for the bulk of BF16 logits; exp(t) = 2^a (1 + c)
// with a = t log2 e rounded and c = t - a ln 2 recovered by two fused
// multiply-adds (the rounding error of a, carried to first order);
// coef = -g (1 - delta) ~ -g exp(-delta) folds g and delta in once per row.
// The target column uses g * (1 - p) = -g * expm1(x - lse).
template <bool kVecIn, bool kVecOut, bool kInPlace>
__global__ void __launch_bounds__(kBwdThreads)
k_logp_bwd(const uint16_t* x, int64_t n, int64_t v, int64_t ld,
           const int64_t* __restrict__ y, int64_t ignore_index, const float* __restrict__ lse,
           const float* __restrict__ g, uint16_t* dx, int64_t ld_out, int64_t segs) {
    const int64_t items = n * segs;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t t = item / segs;
        const int64_t col0 = (item - t * segs) * kBwdSegCols;
        const uint16_t* xr = x + t * ld;
        uint16_t* dr = dx + t * ld_out;
        const int64_t yt = __ldg(y + t);
        const bool act = row_active(yt, v, ignore_index);
        if (!act) {
#pragma unroll
            for (int u = 0; u < kBwdVecPerThread; ++u) {
                const int64_t col = col0 + ((int64_t)u * kBwdThreads + threadIdx.x) * 8;
                if (col >= v) break;
                if (kVecOut && col + 8 <= v) {
                    st_cs_v4(dr + col, make_uint4(0u, 0u, 0u, 0u));
                } else {
                    for (int j = 0; j < 8 && col + j < v; ++j) dr[col + j] = 0;
                }
            }
            continue;
        }
        const float l = __ldg(lse + t);
        const float gt = __ldg(g + t);
        const float lr = (fabsf(l) < 8388608.f) ? __fmul_rn(rintf(__fmul_rn(l, 65536.f)), 1.f / 65536.f) : l;
        const float delta = __fsub_rn(l, lr);          // exact
        const float coef = __fmaf_rn(gt, delta, -gt);   // -g (1 - delta)

        float f[kBwdVecPerThread][8];
#pragma unroll
        for (int u = 0; u < kBwdVecPerThread; ++u) {
            const int64_t col = col0 + ((int64_t)u * kBwdThreads + threadIdx.x) * 8;
            if (kVecIn && col + 8 <= v) {
                const uint4 q = kInPlace ? ld_v4(xr + col) : ld_nc_v4(xr + col);
                f[u][0] = bf_lo(q.x); f[u][1] = bf_hi(q.x);
                f[u][2] = bf_lo(q.y); f[u][3] = bf_hi(q.y);
                f[u][4] = bf_lo(q.z); f[u][5] = bf_hi(q.z);
                f[u][6] = bf_lo(q.w); f[u][7] = bf_hi(q.w);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    f[u][j] = (col + j < v)
                                  ? __uint_as_float((uint32_t)(kInPlace ? xr[col + j]
                                                                         : __ldg(reinterpret_cast<const unsigned short*>(xr + col + j)))
                                                    << 16)
                                  : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kBwdVecPerThread; ++u) {
            const int64_t col = col0 + ((int64_t)u * kBwdThreads + threadIdx.x) * 8;
            if (col >= v) break;
            float d[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // clamped so that a -inf logit gives exp = 0 and a finite c
                const float tt = fmaxf(__fsub_rn(f[u][j], lr), -200.f);
                const float a = __fmul_rn(tt, kLog2e);
                float c = __fmaf_rn(-a, kLn2Hi, tt);
                c = __fmaf_rn(-a, kLn2Lo, c);
                const float q = __fmul_rn(ex2_full(a), coef);
                d[j] = __fmaf_rn(q, c, q);
            }
            const int64_t jt = yt - col;
            if (jt >= 0 && jt < 8) {
                // target column: g * (1 - p) without cancellation
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j == jt) d[j] = __fmul_rn(-gt, expm1f(__fsub_rn(__fsub_rn(f[u][j], lr), delta)));
            }
            if (kVecOut && col + 8 <= v) {
                st_cs_v4(dr + col, make_uint4(pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3]),
                                              pack_bf16x2(d[4], d[5]), pack_bf16x2(d[6], d[7])));
            } else {
                for (int j = 0; j < 8 && col + j < v; ++j)
                    dr[col + j] = (uint16_t)(pack_bf16x2(d[j], 0.f) & 0xffffu);
            }
        }
    }
}

}  // namespace flp
