// Device code of the selected-token log-probability path for sm_103a.
//
// Forward (RL-Kernel issue #241 "TP-aware deterministic logprob", Background
// and PR 3 bullets): LSE_t = log sum_v exp(x[t, v]) with FP32 accumulation,
// logp_t = x[t, y_t] - LSE_t.  Every row is cut into 16 fixed vocabulary tiles
// of width W = 8 * ceil(V / 128); one warp reduces one tile: each lane keeps
// an online (max, sumexp) pair over its fixed share of the tile, the warp
// merges the 32 pairs with a fixed xor butterfly, and a half warp merges the
// 16 tile partials with a fixed pairwise tree in tile-index order (RL-Kernel
// PR #314, Tensor Parallel section: fixed tiles, one fixed merge order).
// Nothing in this order depends on N, on the row's position or on the grid, so
// every row's bits are batch-invariant, and a vocab shard that reduces its own
// tiles with the same functions reproduces the same partials bit for bit.
//
// Backward (RL-Kernel PR #495 "zero-workspace fused backward", Summary item
// 2): dlogits = g * (onehot - exp(x - LSE)) from the saved LSE, one read and
// one write per logit, elementwise.
//
// Arithmetic on pairs uses the packed binary32 instructions of sm_100+
// (add/mul/fma .f32x2, each lane an ordinary IEEE round-to-nearest operation)
// and the packed BF16 maximum; every rounding is explicit, so the full and the
// shard kernels cannot differ by a contraction.  All index arithmetic is
// 64-bit.  The only waits are bounded waits of a warp on its own bulk copies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flp {

constexpr int kTiles = 16;                  // vocabulary tiles per row (K)
constexpr int kWarp = 32;
constexpr int kFwdThreads = kTiles * kWarp; // one warp per tile
constexpr int kGroup = 4;                   // 16-byte vectors per lane per online step
constexpr int kGroupVecs = kWarp * kGroup;  // vectors of a tile per group (128)
constexpr int kStages = 3;                  // bulk-copy ring depth per warp
constexpr int kStageBytes = kGroupVecs * 16;
constexpr int kFwdSmemBytes = kTiles * kStages * kStageBytes + kTiles * kStages * 8;
constexpr int kBwdThreads = 256;
constexpr int kBwdVecPerThread = 4;
constexpr int64_t kBwdSegCols = (int64_t)kBwdThreads * kBwdVecPerThread * 8;
constexpr uint32_t kNegInf2 = 0xff80ff80u;  // two BF16 -inf
// Bounded waits give up after this many SM cycles (about 2 s at 2 GHz).
constexpr long long kWaitLimitCycles = 4000000000LL;

// Mathematical constants: ln 2 to double precision, its binary32 head and
// tail (head + tail = ln 2 to about 2^-48 relative), and log2(e) rounded to
// binary32.
constexpr double kLn2 = 0.6931471805599453094172321214581766;
constexpr float kLn2Hi = (float)kLn2;
constexpr float kLn2Lo = (float)(kLn2 - (double)kLn2Hi);
constexpr float kLog2e = (float)(1.0 / kLn2);

// Sticky device error word: 1 = a bounded wait ran out.  Read and cleared by
// flp_device_error().
__device__ int g_device_error;

struct MS {
    float m;  // running maximum (always the value of an input element, or -inf)
    float s;  // sum of exp(x - m) over the elements seen
};

typedef unsigned long long u64;

// ---------------------------------------------------------------- packed arithmetic

__device__ __forceinline__ u64 f2(float lo, float hi) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(u64 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ u64 f2_add(u64 a, u64 b) {
    u64 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 f2_mul(u64 a, u64 b) {
    u64 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 f2_fma(u64 a, u64 b, u64 c) {
    u64 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// A BF16 value is the top half of a binary32: widening is a shift or a mask.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ u64 bf2_widen(uint32_t w) { return f2(bf_lo(w), bf_hi(w)); }
// (x_lo - b, x_hi - b) for the two BF16 values of w: each widened exactly and
// rounded once (mixed-precision subtract, a BF16 operand and a binary32 one).
__device__ __forceinline__ u64 bf2_sub(uint32_t w, float b) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "sub.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w), "f"(b));
    return f2(lo, hi);
}
__device__ __forceinline__ uint32_t ldg_u16(const uint16_t* p) {
    return (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p));
}
__device__ __forceinline__ float bf_scalar(const uint16_t* p) { return __uint_as_float(ldg_u16(p) << 16); }

// Two binary32 -> packed BF16 pair, round to nearest even (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^a on the special-function unit; results below 2^-126 flush to zero.
__device__ __forceinline__ float ex2_ftz(float a) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// ---------------------------------------------------------------- memory access

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
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr)
                 : "memory");
    return r;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// mbarrier and bulk-copy (TMA, non-tensor) primitives.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// One probe of phase `parity` of an mbarrier.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Wait for phase `parity` of an mbarrier, giving up after `limit` cycles.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 31u) == 0 && clock64() - t0 > limit) return false;
    }
}

// ---------------------------------------------------------------- forward reduction

// One online step of a lane over kGroup vectors of 8 BF16 (q[u] = the four
// 32-bit words of vector u; with kFull all vectors hold data, otherwise
// vectors [0, nvalid) do and the others are -inf): gm = max(m, elements) by
// packed BF16 maxima; each element's term 2^((x - gm) log2 e) on the
// special-function unit (x - gm is exact: both are BF16 values); the terms
// summed by a fixed pairwise tree (word pairs, then vectors:
// ((w0 + w1) + (w2 + w3)) lane-wise, vectors ((v0 + v1) + (v2 + v3)), then the
// even and odd lanes); s = s * exp(m - gm) + group sum.
template <bool kFull>
__device__ __forceinline__ void group_update(const uint32_t (&q)[kGroup][4], int nvalid, float& m,
                                             float& s) {
    uint32_t w = bf2_max(bf2_max(q[0][0], q[0][1]), bf2_max(q[0][2], q[0][3]));
#pragma unroll
    for (int u = 1; u < kGroup; ++u)
        w = bf2_max(w, bf2_max(bf2_max(q[u][0], q[u][1]), bf2_max(q[u][2], q[u][3])));
    const float gm = fmaxf(m, fmaxf(bf_lo(w), bf_hi(w)));
    if (gm == -INFINITY) return;  // nothing finite seen yet: (m, s) stays (-inf, 0)
    const u64 l2e = f2(kLog2e, kLog2e);
    u64 vsum[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
        if (kFull || u < nvalid) {
            u64 p[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float a0, a1;
                f2_split(f2_mul(bf2_sub(q[u][k], gm), l2e), a0, a1);
                p[k] = f2(ex2_ftz(a0), ex2_ftz(a1));
            }
            vsum[u] = f2_add(f2_add(p[0], p[1]), f2_add(p[2], p[3]));
        } else {
            vsum[u] = 0ull;
        }
    }
    static_assert(kGroup == 4, "the group tree is written for four vectors");
    float e, o;
    f2_split(f2_add(f2_add(vsum[0], vsum[1]), f2_add(vsum[2], vsum[3])), e, o);
    const float gs = __fadd_rn(e, o);
    const float r = (m == gm) ? 1.f : ex2_ftz(__fmul_rn(__fsub_rn(m, gm), kLog2e));
    s = __fmaf_rn(s, r, gs);
    m = gm;
}

// The four words of the 8 columns [col, col + 8) of a tile; columns >= width
// read as -inf (padded columns are masked, PR #314 ReductionSpec).  The vector
// path needs a 16-byte aligned tile; both paths give the same words.
template <bool kVec>
__device__ __forceinline__ void load_words(const uint16_t* __restrict__ tile, int64_t col,
                                           int64_t width, uint32_t (&w)[4]) {
    if (kVec && col + 8 <= width) {
        const uint4 q = ld_nc_v4(tile + col);
        w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = (col + 2 * k < width) ? ldg_u16(tile + col + 2 * k) : 0xff80u;
            const uint32_t hi = (col + 2 * k + 1 < width) ? ldg_u16(tile + col + 2 * k + 1) : 0xff80u;
            w[k] = lo | (hi << 16);
        }
    }
}

// Online (max, sumexp) of one lane over a tile of `width` columns: 16-byte
// vector j of the tile belongs to lane j mod 32, and the lane visits its
// vectors in increasing j, kGroup at a time (vectors v0 + 32u + lane of group
// v0 / 128).  Plain loads; the bulk-copy forward feeds group_update with the
// same words in the same order.
template <bool kVec>
__device__ __forceinline__ MS tile_scan(const uint16_t* __restrict__ tile, int64_t width,
                                        int lane) {
    const int64_t nvec = (width + 7) >> 3;
    float m = -INFINITY, s = 0.f;
    for (int64_t v0 = 0; v0 < nvec; v0 += kGroupVecs) {
        uint32_t q[kGroup][4];
        int nvalid = 0;
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int64_t j = v0 + (int64_t)kWarp * u + lane;
            if (j < nvec) {
                load_words<kVec>(tile, j * 8, width, q[u]);
                nvalid = u + 1;
            } else {
                q[u][0] = q[u][1] = q[u][2] = q[u][3] = kNegInf2;
            }
        }
        if (nvalid == kGroup) group_update<true>(q, nvalid, m, s);
        else group_update<false>(q, nvalid, m, s);
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
// (lane k of the half holds tile k; tiles beyond the vocabulary hold the
// identity (-inf, 0)).  M = max m_k; S = sum_k s_k exp(m_k - M) summed as a
// fixed pairwise tree in tile-index order (issue #241 PR 3 merge formula).
// m_k - M is exact; exp is the accurate library expf.  All 32 lanes call this
// together; every lane gets (M, S) of its half.
__device__ __forceinline__ MS tile_fold16(MS p) {
    float M = p.m;
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off, 16));
    float term = (p.m == -INFINITY) ? 0.f : __fmul_rn(p.s, expf(__fsub_rn(p.m, M)));
#pragma unroll
    for (int off = 1; off <= 8; off <<= 1)
        term = __fadd_rn(term, __shfl_xor_sync(0xffffffffu, term, off, 16));
    return MS{M, term};
}

// LSE = M + log S and logp = x_y - LSE, the log and the subtractions carried
// in double and each output rounded once to binary32 (the "downcast at final
// write" of issue #241 Goal).  lse_lo, when given, receives the binary32
// rounding residual of the LSE (LSE - lse), so that lse + lse_lo carries the
// LSE to about 2^-48 relative for the backward.
__device__ __forceinline__ void finalize_row(MS f, bool active, float x_y, float* logp_out,
                                             float* lse_out, float* lse_lo_out) {
    const double l = (f.m == -INFINITY) ? -(double)INFINITY : (double)f.m + log((double)f.s);
    const float lf = __double2float_rn(l);
    *lse_out = lf;
    if (lse_lo_out) *lse_lo_out = isfinite(lf) ? __double2float_rn(l - (double)lf) : 0.f;
    *logp_out = active ? __double2float_rn((double)x_y - l) : 0.f;
}

__device__ __forceinline__ bool row_active(int64_t y, int64_t v, int64_t ignore_index) {
    return y >= 0 && y < v && y != ignore_index;
}

// ---------------------------------------------------------------- forward kernels

// Forward with plain loads (any alignment): one CTA of 16 warps per row, warp
// k reduces tile k.
template <bool kVec>
__global__ void __launch_bounds__(kFwdThreads)
k_logp_fwd(const uint16_t* __restrict__ x, int64_t n, int64_t v, int64_t ld, int64_t W,
           const int64_t* __restrict__ y, int64_t ignore_index, float* __restrict__ logp,
           float* __restrict__ lse, float* __restrict__ lse_lo) {
    __shared__ float sh_m[kTiles], sh_s[kTiles];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
        const uint16_t* __restrict__ xr = x + t * ld;
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
            const MS f = tile_fold16(MS{sh_m[k], sh_s[k]});
            if (lane == 0) finalize_row(f, act, x_y, logp + t, lse + t, lse_lo ? lse_lo + t : nullptr);
        }
        __syncthreads();
    }
}

// Forward with bulk copies (16-byte aligned rows, ld % 8 == 0, V < 2^31).
// Persistent CTAs of 16 warps; CTA b takes rows b, b + grid, b + 2 grid, ...
// Each warp streams its tile of successive rows through a private ring of
// kStages shared-memory stages (one 2 KB group each): lane 0 issues
// cp.async.bulk for group i + kStages as soon as the warp has read group i,
// so copies of the next row are already in flight while a row is finished.
// The lanes read the same words, in the same order, as tile_scan would load
// them (a ragged last vector is read from global memory), so results are
// bitwise those of k_logp_fwd.  Tile partials go to a double-buffered shared
// array; after one barrier per row, warp (row mod 16) merges them and writes
// the row.  A wait that runs out sets g_device_error; the warp then stops
// issuing copies and skips waits, and drains its copies in flight before
// exiting.
__global__ void __launch_bounds__(kFwdThreads, 2)
k_logp_fwd_bulk(const uint16_t* __restrict__ x, int64_t n, int64_t v, int64_t ld, int64_t W,
                const int64_t* __restrict__ y, int64_t ignore_index, float* __restrict__ logp,
                float* __restrict__ lse, float* __restrict__ lse_lo) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float sh_m[2][kTiles], sh_s[2][kTiles];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t stage0 = smem_u32(smem + warp * kStages * kStageBytes);
    const uint32_t bar0 = smem_u32(smem + kTiles * kStages * kStageBytes) + warp * kStages * 8;
    if (threadIdx.x < kTiles * kStages)
        mbar_init(smem_u32(smem + kTiles * kStages * kStageBytes) + threadIdx.x * 8, 1);
    fence_mbar_init();
    __syncthreads();

    // tile-local extents fit in 32 bits (the host routes V >= 2^31 elsewhere)
    const int64_t c0 = (int64_t)warp * W;
    const int width = (int)(c0 >= v ? 0 : (v - c0 < W ? v - c0 : W));
    const int nfull = width >> 3, nvec = (width + 7) >> 3;
    const int G = (nvec + kGroupVecs - 1) / kGroupVecs;          // groups per row
    const int Gfull = nfull / kGroupVecs;                        // groups of 128 full vectors
    const int64_t rows = (n > (int64_t)blockIdx.x) ? (n - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t jobs = rows * G;
    const int64_t row_step = (int64_t)gridDim.x * ld;

    // Issuer: group iss_g of the row at iss_row (its first element of this
    // tile), stage iss_st.  Every lane tracks it; lane 0 issues.
    const uint16_t* iss_row = x + (int64_t)blockIdx.x * ld + c0;
    int iss_g = 0, iss_st = 0;
    int64_t issued = 0;
    auto issue_next = [&]() {
        if (lane == 0) {
            const int nv = nfull - iss_g * kGroupVecs;
            const uint32_t bytes = nv <= 0 ? 0u : (uint32_t)((nv < kGroupVecs ? nv : kGroupVecs) * 16);
            const uint32_t bar = bar0 + iss_st * 8;
            mbar_arrive_expect_tx(bar, bytes);
            if (bytes) bulk_g2s(stage0 + iss_st * kStageBytes, iss_row + iss_g * (kGroupVecs * 8), bytes, bar);
        }
        if (++iss_g == G) {
            iss_g = 0;
            iss_row += row_step;
        }
        if (++iss_st == kStages) iss_st = 0;
        ++issued;
    };

    bool ok = true;
    int64_t fail_at = -1;
    while (issued < kStages && issued < jobs) issue_next();

    int st = 0;          // stage of the next group to consume
    uint32_t phase = 0;  // its mbarrier parity
    for (int64_t j = 0; j < rows; ++j) {
        const int64_t t = (int64_t)blockIdx.x + j * gridDim.x;
        const int folder = (int)(j % kTiles);
        bool act = false;
        float x_y = 0.f;
        if (warp == folder && lane == 0) {
            const int64_t yt = __ldg(y + t);
            act = row_active(yt, v, ignore_index);
            if (act) x_y = bf_scalar(x + t * ld + yt);
        }
        const uint16_t* __restrict__ tile = x + t * ld + c0;
        float m = -INFINITY, s = 0.f;
        for (int g = 0; g < G; ++g) {
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar0 + st * 8, phase, kWaitLimitCycles));
                if (!ok) fail_at = j * G + g;
            }
            const uint32_t sbase = stage0 + st * kStageBytes + lane * 16;
            uint32_t q[kGroup][4];
            if (g < Gfull) {
#pragma unroll
                for (int u = 0; u < kGroup; ++u) {
                    const uint4 r = lds_v4(sbase + u * (kWarp * 16));
                    q[u][0] = r.x; q[u][1] = r.y; q[u][2] = r.z; q[u][3] = r.w;
                }
                __syncwarp();
                if (ok && issued < jobs) {
                    if (lane == 0) fence_proxy_async_smem();
                    issue_next();
                }
                group_update<true>(q, kGroup, m, s);
            } else {
                const int v0 = g * kGroupVecs;
                int nvalid = 0;
#pragma unroll
                for (int u = 0; u < kGroup; ++u) {
                    const int jv = v0 + kWarp * u + lane;
                    if (jv < nfull) {
                        const uint4 r = lds_v4(sbase + u * (kWarp * 16));
                        q[u][0] = r.x; q[u][1] = r.y; q[u][2] = r.z; q[u][3] = r.w;
                        nvalid = u + 1;
                    } else if (jv < nvec) {
                        load_words<false>(tile, (int64_t)jv * 8, width, q[u]);
                        nvalid = u + 1;
                    } else {
                        q[u][0] = q[u][1] = q[u][2] = q[u][3] = kNegInf2;
                    }
                }
                __syncwarp();
                if (ok && issued < jobs) {
                    if (lane == 0) fence_proxy_async_smem();
                    issue_next();
                }
                if (nvalid == kGroup) group_update<true>(q, nvalid, m, s);
                else group_update<false>(q, nvalid, m, s);
            }
            if (++st == kStages) {
                st = 0;
                phase ^= 1u;
            }
        }
        MS p = warp_merge(MS{m, s});
        if (lane == 0) {
            sh_m[j & 1][warp] = p.m;
            sh_s[j & 1][warp] = p.s;
        }
        __syncthreads();
        if (warp == folder) {
            const int k = lane & 15;
            const MS f = tile_fold16(MS{sh_m[j & 1][k], sh_s[j & 1][k]});
            if (lane == 0) finalize_row(f, act, x_y, logp + t, lse + t, lse_lo ? lse_lo + t : nullptr);
        }
    }
    if (!ok) {
        if (lane == 0) atomicExch(&g_device_error, 1);
        // drain the copies issued but never waited for (at most kStages)
        for (int64_t k = fail_at; k < issued; ++k)
            (void)mbar_wait(bar0 + (int)(k % kStages) * 8, (uint32_t)((k / kStages) & 1), kWaitLimitCycles);
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
             float* __restrict__ logp, float* __restrict__ lse, float* __restrict__ lse_lo) {
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
        const MS f = tile_fold16(p);
        if (valid && k == 0) {
            const int64_t yt = __ldg(y + t);
            const bool act = row_active(yt, v, ignore_index);
            const float x_y = act ? __ldg(sel + t) : 0.f;
            finalize_row(f, act, x_y, logp + t, lse + t, lse_lo ? lse_lo + t : nullptr);
        }
    }
}

// ---------------------------------------------------------------- backward

// Per-row constants of the backward (see k_logp_bwd).
struct BwdRow {
    u64 neg_lr;   // (-lse_r, -lse_r)
    u64 coef2;    // (coef, coef), coef = -g (1 - delta)
    uint32_t floor_w;
    float lr, delta, g;
};

// Gradient of one vector of 8 columns (words w, output words o), target
// column jt (or outside [0, 8)).
__device__ __forceinline__ void bwd_vector(const uint32_t (&w)[4], const BwdRow& r, int64_t jt,
                                           uint32_t (&o)[4]) {
    const u64 l2e = f2(kLog2e, kLog2e);
    const u64 nln2hi = f2(-kLn2Hi, -kLn2Hi), nln2lo = f2(-kLn2Lo, -kLn2Lo);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const u64 tt = f2_add(bf2_widen(bf2_max(w[k], r.floor_w)), r.neg_lr);
        const u64 a = f2_mul(tt, l2e);
        const u64 c = f2_fma(a, nln2lo, f2_fma(a, nln2hi, tt));
        float a0, a1;
        f2_split(a, a0, a1);
        const u64 q = f2_mul(f2(ex2_ftz(a0), ex2_ftz(a1)), r.coef2);
        float d0, d1;
        f2_split(f2_fma(q, c, q), d0, d1);
        o[k] = pack_bf16x2(d0, d1);
    }
    if (jt >= 0 && jt < 8) {
        // target column: g * (1 - p) without cancellation
        const int kt = (int)(jt >> 1);
        uint32_t wk = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k == kt) wk = w[k];
        wk = bf2_max(wk, r.floor_w);
        const float xt = (jt & 1) ? bf_hi(wk) : bf_lo(wk);
        const float dt = __fmul_rn(-r.g, expm1f(__fsub_rn(__fsub_rn(xt, r.lr), r.delta)));
        const uint32_t bt = pack_bf16x2(dt, dt) & 0xffffu;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k == kt) o[k] = (jt & 1) ? ((o[k] & 0xffffu) | (bt << 16)) : ((o[k] & 0xffff0000u) | bt);
    }
}

template <bool kVecIn, bool kInPlace>
__device__ __forceinline__ void bwd_load(const uint16_t* xr, int64_t col, int64_t v, uint32_t (&w)[4]) {
    if (kVecIn && col + 8 <= v) {
        const uint4 q = kInPlace ? ld_v4(xr + col) : ld_nc_v4(xr + col);
        w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t lo = 0, hi = 0;
            if (col + 2 * k < v) lo = kInPlace ? xr[col + 2 * k] : ldg_u16(xr + col + 2 * k);
            if (col + 2 * k + 1 < v) hi = kInPlace ? xr[col + 2 * k + 1] : ldg_u16(xr + col + 2 * k + 1);
            w[k] = lo | (hi << 16);
        }
    }
}

template <bool kVecOut>
__device__ __forceinline__ void bwd_store(uint16_t* dr, int64_t col, int64_t v, const uint32_t (&o)[4]) {
    if (kVecOut && col + 8 <= v) {
        st_cs_v4(dr + col, make_uint4(o[0], o[1], o[2], o[3]));
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (col + j < v) dr[col + j] = (uint16_t)((j & 1) ? (o[j >> 1] >> 16) : (o[j >> 1] & 0xffffu));
    }
}

// Backward: one CTA per (row, segment of kBwdSegCols columns), elementwise.
// Per active row: LSE = lse (+ lse_lo) is split as lse_r + delta with lse_r
// on a 2^-16 grid, so that t = x - lse_r is exact for the bulk of BF16
// logits; exp(t) = 2^a (1 + c) with a = t log2 e rounded and c = t - a ln 2
// recovered by two fused multiply-adds against a two-float ln 2 (the rounding
// error of a, carried to first order); coef = -g (1 - delta) ~ -g exp(-delta)
// folds g and delta in once per row.  Logits below LSE - 200 are raised to
// that bound first (their exp is below 2^-288, zero in binary32), which also
// keeps a -inf logit from producing inf - inf.  The target column is
// g * (1 - p) = -g * expm1(x - LSE), without cancellation.  Values below
// 2^-126 flush to zero.  Each thread loads its four vectors before computing
// any, so four 16-byte loads are in flight per thread.
template <bool kVecIn, bool kVecOut, bool kInPlace>
__global__ void __launch_bounds__(kBwdThreads)
k_logp_bwd(const uint16_t* x, int64_t n, int64_t v, int64_t ld, const int64_t* __restrict__ y,
           int64_t ignore_index, const float* __restrict__ lse, const float* __restrict__ lse_lo,
           const float* __restrict__ g, uint16_t* dx, int64_t ld_out, int64_t segs) {
    const int64_t items = n * segs;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t t = item / segs;
        const int64_t col0 = (item - t * segs) * kBwdSegCols + (int64_t)threadIdx.x * 8;
        const uint16_t* xr = x + t * ld;
        uint16_t* dr = dx + t * ld_out;
        const int64_t yt = __ldg(y + t);
        if (!row_active(yt, v, ignore_index)) {
            const uint32_t z[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int u = 0; u < kBwdVecPerThread; ++u) {
                const int64_t col = col0 + (int64_t)u * kBwdThreads * 8;
                if (col < v) bwd_store<kVecOut>(dr, col, v, z);
            }
            continue;
        }
        BwdRow r;
        const float l = __ldg(lse + t);
        const float l_lo = lse_lo ? __ldg(lse_lo + t) : 0.f;
        r.g = __ldg(g + t);
        r.lr = (fabsf(l) < 8388608.f) ? __fmul_rn(rintf(__fmul_rn(l, 65536.f)), 1.f / 65536.f) : l;
        r.delta = __fadd_rn(__fsub_rn(l, r.lr), l_lo);          // l - lr is exact
        const float coef = __fmaf_rn(r.g, r.delta, -r.g);        // -g (1 - delta)
        r.floor_w = kNegInf2;
        if (fabsf(l) < 1048576.f) {
            const uint32_t b = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rd(__fsub_rn(l, 200.f)));
            r.floor_w = b | (b << 16);
        }
        r.neg_lr = f2(-r.lr, -r.lr);
        r.coef2 = f2(coef, coef);

        uint32_t w0[4], w1[4], w2[4], w3[4];
        static_assert(kBwdVecPerThread == 4, "four vectors per thread");
        const int64_t cs = (int64_t)kBwdThreads * 8;
        if (col0 < v) bwd_load<kVecIn, kInPlace>(xr, col0, v, w0);
        if (col0 + cs < v) bwd_load<kVecIn, kInPlace>(xr, col0 + cs, v, w1);
        if (col0 + 2 * cs < v) bwd_load<kVecIn, kInPlace>(xr, col0 + 2 * cs, v, w2);
        if (col0 + 3 * cs < v) bwd_load<kVecIn, kInPlace>(xr, col0 + 3 * cs, v, w3);
        uint32_t o[4];
        if (col0 < v) { bwd_vector(w0, r, yt - col0, o); bwd_store<kVecOut>(dr, col0, v, o); }
        if (col0 + cs < v) { bwd_vector(w1, r, yt - (col0 + cs), o); bwd_store<kVecOut>(dr, col0 + cs, v, o); }
        if (col0 + 2 * cs < v) { bwd_vector(w2, r, yt - (col0 + 2 * cs), o); bwd_store<kVecOut>(dr, col0 + 2 * cs, v, o); }
        if (col0 + 3 * cs < v) { bwd_vector(w3, r, yt - (col0 + 3 * cs), o); bwd_store<kVecOut>(dr, col0 + 3 * cs, v, o); }
    }
}

// Result word of the bounded-wait self-test.
__device__ int g_selftest_result;

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives on, with a short cycle limit, and records whether the wait gave up.
__global__ void k_wait_timeout_selftest(long long limit) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const bool done = mbar_wait(b, 0, limit);
    g_selftest_result = done ? 0 : 1;
    if (!done) atomicExch(&g_device_error, 1);
}

}  // namespace flp
