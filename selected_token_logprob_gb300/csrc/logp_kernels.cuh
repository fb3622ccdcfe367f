// Device code of the selected-token log-probability path for sm_103a.
//
// Forward (RL-Kernel issue #241 "TP-aware deterministic logprob", Background
// and PR 3 bullets): LSE_t = log sum_v exp(s x[t, v]) with FP32 accumulation,
// logp_t = s x[t, y_t] - LSE_t, where s = 1/T is the inverse temperature
// (s = 1 unless rollout logprobs at a temperature are asked for, PR #495
// provider experiment).  Every row is cut into 16 fixed vocabulary tiles of
// width W = 8 * ceil(V / 128); one warp reduces one tile: each lane keeps an
// online (max, sumexp) pair over its fixed share of the tile, the warp merges
// the 32 pairs with a fixed xor butterfly, and a half warp merges the 16 tile
// partials with a fixed pairwise tree in tile-index order (RL-Kernel PR #314,
// Tensor Parallel section: fixed tiles, one fixed merge order).  Nothing in
// this order depends on N, on the row's position or on the grid, so every
// row's bits are batch-invariant, and a vocab shard that reduces its own tiles
// with the same functions reproduces the same partials bit for bit.
//
// Backward (RL-Kernel PR #495 "zero-workspace fused backward", Summary item
// 2): dlogits = s g (onehot - exp(s x - LSE)) from the saved LSE, one read
// and one write per logit, elementwise, written in the logits' dtype.
//
// Logits may be BF16, FP16 or FP32 (PR #495 Tests: FP32/BF16/FP16).  A
// "unit" is 8 consecutive elements of a row (16 bytes for 16-bit types, 32 for
// FP32); lane j of a warp owns units j, j + 32, ... of its tile.  Rows may be
// excluded by an explicit active mask (PR #314, MaskMode).  All index
// arithmetic is 64-bit except tile-local indices of the bulk forward.  The
// only waits are bounded waits of a warp on its own bulk copies.
#pragma once

#include "logp_prims.cuh"

namespace flp {

enum class Dt : int { BF16 = 0, F16 = 1, F32 = 2 };

constexpr int kTiles = 16;                   // vocabulary tiles per row (K)
constexpr int kWarp = 32;
constexpr int kFwdThreads = kTiles * kWarp;  // one warp per tile
constexpr int kGroup = 4;                    // units per lane per online step
constexpr int kGroupUnits = kWarp * kGroup;  // units of a tile per group (128)
constexpr int kStages = 3;                   // bulk-copy ring depth per warp
constexpr int kBwdThreads = 128;
constexpr int kBwdUnitsPerThread = 8;
constexpr int64_t kBwdSegCols = (int64_t)kBwdThreads * kBwdUnitsPerThread * 8;
// Bounded waits give up after this many SM cycles (about 2 s at 2 GHz).
constexpr long long kWaitLimitCycles = 4000000000LL;

// Mathematical constants: ln 2 to double precision, its binary32 head and
// tail (head + tail = ln 2 to about 2^-48 relative), and log2(e) rounded to
// binary32.
constexpr double kLn2 = 0.6931471805599453094172321214581766;
constexpr float kLn2Hi = (float)kLn2;
constexpr float kLn2Lo = (float)(kLn2 - (double)kLn2Hi);
constexpr float kLog2e = (float)(1.0 / kLn2);

// Mean relative error of ex2.approx.ftz.f32 on this GPU family: -4.95e-8
// (measured over 4M arguments in [-24, 0]; flat in the argument; re-measured
// by flp_selftest_ex2_bias).  Every tile sum is built from such terms, so it
// is scaled by (1 + kEx2BiasComp) once, in tile_partial.
constexpr float kEx2BiasComp = 4.95e-8f;

// Sticky device error word: 1 = a bounded wait ran out.  Read and cleared by
// flp_device_error().
__device__ int g_device_error;

struct MS {
    float m;  // running maximum of the raw logits (an input element, or -inf)
    float s;  // sum of exp(s (x - m)) over the elements seen
};

// Inverse temperature s and s log2(e) as a two-float (hi + lo).
struct Scale {
    float s, hi, lo;
};

// ---------------------------------------------------------------- units by dtype

template <Dt D>
struct Unit {
    static constexpr int kWords = (D == Dt::F32) ? 8 : 4;
    static constexpr int kBytes = kWords * 4;
    static constexpr int kElemBytes = (D == Dt::F32) ? 4 : 2;
    static constexpr uint32_t kNegInfBits = (D == Dt::BF16) ? 0xff80u : (D == Dt::F16) ? 0xfc00u : 0xff800000u;
    uint32_t w[kWords];
};

template <Dt D>
constexpr int kStageBytes = kGroupUnits * Unit<D>::kBytes;
template <Dt D>
constexpr int kFwdSmemBytes = kTiles * kStages * kStageBytes<D> + kTiles * kStages * 8;
template <Dt D>
constexpr int kFwdMinBlocks = (D == Dt::F32) ? 1 : 2;
// backward CTAs of 128 threads per SM: register caps 64 (16-bit) and 96 (FP32)
template <Dt D>
constexpr int kBwdMinBlocks = (D == Dt::F32) ? 5 : 8;

template <Dt D>
__device__ __forceinline__ uint32_t elem_bits(const void* base, int64_t i) {
    if constexpr (D == Dt::F32) return __ldg(reinterpret_cast<const unsigned int*>(base) + i);
    else return (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(base) + i);
}
template <Dt D>
__device__ __forceinline__ uint32_t elem_bits_plain(const void* base, int64_t i) {
    if constexpr (D == Dt::F32) return reinterpret_cast<const unsigned int*>(base)[i];
    else return (uint32_t)reinterpret_cast<const unsigned short*>(base)[i];
}
template <Dt D>
__device__ __forceinline__ float bits_value(uint32_t b) {
    if constexpr (D == Dt::BF16) return __uint_as_float(b << 16);
    else if constexpr (D == Dt::F16) return __half2float(__ushort_as_half((unsigned short)b));
    else return __uint_as_float(b);
}
template <Dt D>
__device__ __forceinline__ float elem_value(const void* base, int64_t i) {
    return bits_value<D>(elem_bits<D>(base, i));
}

template <Dt D>
__device__ __forceinline__ void unit_fill_neg_inf(Unit<D>& u) {
    constexpr uint32_t w = (D == Dt::F32) ? Unit<D>::kNegInfBits : (Unit<D>::kNegInfBits * 0x10001u);
#pragma unroll
    for (int k = 0; k < Unit<D>::kWords; ++k) u.w[k] = w;
}

// The unit of the 8 columns [col, col + 8) of a tile; columns >= width read
// as -inf (padded columns are masked, PR #314 ReductionSpec).  The vector path
// needs a 16-byte aligned tile; both paths give the same words.
template <Dt D, bool kVec>
__device__ __forceinline__ void unit_load(const void* __restrict__ tile, int64_t col, int64_t width,
                                          Unit<D>& u) {
    constexpr uint32_t NI = Unit<D>::kNegInfBits;
    if (kVec && col + 8 <= width) {
        const char* p = reinterpret_cast<const char*>(tile) + col * Unit<D>::kElemBytes;
        const uint4 a = ld_nc_v4(p);
        u.w[0] = a.x; u.w[1] = a.y; u.w[2] = a.z; u.w[3] = a.w;
        if constexpr (D == Dt::F32) {
            const uint4 b = ld_nc_v4(p + 16);
            u.w[4] = b.x; u.w[5] = b.y; u.w[6] = b.z; u.w[7] = b.w;
        }
    } else if constexpr (D == Dt::F32) {
#pragma unroll
        for (int j = 0; j < 8; ++j) u.w[j] = (col + j < width) ? elem_bits<D>(tile, col + j) : NI;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = (col + 2 * k < width) ? elem_bits<D>(tile, col + 2 * k) : NI;
            const uint32_t hi = (col + 2 * k + 1 < width) ? elem_bits<D>(tile, col + 2 * k + 1) : NI;
            u.w[k] = lo | (hi << 16);
        }
    }
}

template <Dt D>
__device__ __forceinline__ void unit_load_shared(uint32_t addr, Unit<D>& u) {
    const uint4 a = lds_v4(addr);
    u.w[0] = a.x; u.w[1] = a.y; u.w[2] = a.z; u.w[3] = a.w;
    if constexpr (D == Dt::F32) {
        const uint4 b = lds_v4(addr + 16);
        u.w[4] = b.x; u.w[5] = b.y; u.w[6] = b.z; u.w[7] = b.w;
    }
}

// max(m, all elements of the group's units), by packed 16-bit maxima.
template <Dt D>
__device__ __forceinline__ float group_max(const Unit<D> (&q)[kGroup], float m) {
    if constexpr (D == Dt::F32) {
        float r = m;
#pragma unroll
        for (int u = 0; u < kGroup; ++u)
#pragma unroll
            for (int j = 0; j < 8; ++j) r = fmaxf(r, __uint_as_float(q[u].w[j]));
        return r;
    } else {
        auto mx = [](uint32_t a, uint32_t b) { return D == Dt::BF16 ? bf2_max(a, b) : h2_max(a, b); };
        uint32_t w = mx(mx(q[0].w[0], q[0].w[1]), mx(q[0].w[2], q[0].w[3]));
#pragma unroll
        for (int u = 1; u < kGroup; ++u) w = mx(w, mx(mx(q[u].w[0], q[u].w[1]), mx(q[u].w[2], q[u].w[3])));
        const float lo = (D == Dt::BF16) ? bf_lo(w) : h_lo(w);
        const float hi = (D == Dt::BF16) ? bf_hi(w) : h_hi(w);
        return fmaxf(m, fmaxf(lo, hi));
    }
}

// (x_{2k} - b, x_{2k+1} - b) of a unit, each rounded once.
template <Dt D>
__device__ __forceinline__ u64 pair_sub(const Unit<D>& u, int k, float b) {
    if constexpr (D == Dt::BF16) return bf2_sub(u.w[k], b);
    else if constexpr (D == Dt::F16) return h2_sub(u.w[k], b);
    else return f2_add(f2(__uint_as_float(u.w[2 * k]), __uint_as_float(u.w[2 * k + 1])), f2(-b, -b));
}

// t log2(e) s: one product when s = 1, else against the two-float s log2(e).
template <bool kScaled>
__device__ __forceinline__ u64 to_log2(u64 t, const Scale& sc) {
    if constexpr (kScaled) return f2_fma(t, f2(sc.hi, sc.hi), f2_mul(t, f2(sc.lo, sc.lo)));
    else return f2_mul(t, f2(kLog2e, kLog2e));
}
template <bool kScaled>
__device__ __forceinline__ float to_log2_1(float t, const Scale& sc) {
    if constexpr (kScaled) return __fmaf_rn(t, sc.hi, __fmul_rn(t, sc.lo));
    else return __fmul_rn(t, kLog2e);
}

// ---------------------------------------------------------------- forward reduction

// One online step of a lane over kGroup units (with kFull all hold data,
// otherwise units [0, nvalid) do and the others are -inf).  Maxima are kept in
// units of the raw logits x; the scale enters only the exponent:
// gm = max(m, elements); each element's term 2^((x - gm) s log2 e) on the
// special-function unit (x - gm is exact for 16-bit inputs); the terms summed
// by a fixed pairwise tree (element pairs ((p0 + p1) + (p2 + p3)) lane-wise,
// units ((u0 + u1) + (u2 + u3)), then the even and odd lanes);
// s_acc = s_acc * exp(s (m - gm)) + group sum.
template <Dt D, bool kFull, bool kScaled>
__device__ __forceinline__ void group_update(const Unit<D> (&q)[kGroup], int nvalid, float& m,
                                             float& s, const Scale& sc) {
    const float gm = group_max<D>(q, m);
    if (gm == -INFINITY) return;  // nothing finite seen yet: (m, s) stays (-inf, 0)
    u64 vsum[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
        if (kFull || u < nvalid) {
            u64 p[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float a0, a1;
                f2_split(to_log2<kScaled>(pair_sub<D>(q[u], k, gm), sc), a0, a1);
                p[k] = f2(ex2_ftz(a0), ex2_ftz(a1));
            }
            vsum[u] = f2_add(f2_add(p[0], p[1]), f2_add(p[2], p[3]));
        } else {
            vsum[u] = 0ull;
        }
    }
    static_assert(kGroup == 4, "the group tree is written for four units");
    float e, o;
    f2_split(f2_add(f2_add(vsum[0], vsum[1]), f2_add(vsum[2], vsum[3])), e, o);
    const float gs = __fadd_rn(e, o);
    const float r = (m == gm) ? 1.f : ex2_ftz(to_log2_1<kScaled>(__fsub_rn(m, gm), sc));
    s = __fmaf_rn(s, r, gs);
    m = gm;
}

// Online (max, sumexp) of one lane over a tile of `width` columns with plain
// loads: unit j of the tile belongs to lane j mod 32, visited in increasing j,
// kGroup at a time (units v0 + 32u + lane of group v0 / 128).  The bulk-copy
// forward feeds group_update with the same words in the same order.
template <Dt D, bool kVec, bool kScaled>
__device__ __forceinline__ MS tile_scan(const void* __restrict__ tile, int64_t width, int lane,
                                        const Scale& sc) {
    const int64_t nunit = (width + 7) >> 3;
    float m = -INFINITY, s = 0.f;
    for (int64_t v0 = 0; v0 < nunit; v0 += kGroupUnits) {
        Unit<D> q[kGroup];
        int nvalid = 0;
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int64_t j = v0 + (int64_t)kWarp * u + lane;
            if (j < nunit) {
                unit_load<D, kVec>(tile, j * 8, width, q[u]);
                nvalid = u + 1;
            } else {
                unit_fill_neg_inf<D>(q[u]);
            }
        }
        if (nvalid == kGroup) group_update<D, true, kScaled>(q, nvalid, m, s, sc);
        else group_update<D, false, kScaled>(q, nvalid, m, s, sc);
    }
    return MS{m, s};
}

// Merge of two (max, sumexp) pairs: the pair holding the larger max keeps its
// sum, the other is scaled by exp(s (m_small - M)).  Symmetric in its
// arguments (IEEE addition commutes), so both lanes of a butterfly get the
// same bits.
template <bool kScaled>
__device__ __forceinline__ MS ms_merge(MS a, MS b, const Scale& sc) {
    const bool a_big = a.m >= b.m;
    const float M = a_big ? a.m : b.m;
    const float m_small = a_big ? b.m : a.m;
    const float s_big = a_big ? a.s : b.s;
    const float s_small = a_big ? b.s : a.s;
    float r;
    if (m_small == -INFINITY) r = 0.f;
    else if (m_small == M) r = 1.f;
    else r = ex2_ftz(to_log2_1<kScaled>(__fsub_rn(m_small, M), sc));
    return MS{M, __fmaf_rn(s_small, r, s_big)};
}

// Fixed xor butterfly over the 32 lanes of a warp (offsets 16, 8, 4, 2, 1);
// every lane ends with the same pair.
template <bool kScaled>
__device__ __forceinline__ MS warp_merge(MS p, const Scale& sc) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        MS o;
        o.m = __shfl_xor_sync(0xffffffffu, p.m, off);
        o.s = __shfl_xor_sync(0xffffffffu, p.s, off);
        p = ms_merge<kScaled>(p, o, sc);
    }
    return p;
}

// The partial of a whole tile: the warp butterfly of the lane pairs, with the
// sum corrected for the mean bias of the special-function unit's exp2 (one
// fused multiply-add).  Every path (forward, plain forward, shard partials)
// forms tile partials here, so they stay bitwise equal.
template <bool kScaled>
__device__ __forceinline__ MS tile_partial(MS lane_pair, const Scale& sc) {
    MS p = warp_merge<kScaled>(lane_pair, sc);
    p.s = __fmaf_rn(p.s, kEx2BiasComp, p.s);
    return p;
}

// Merge of the 16 tile partials of one row held by a 16-lane half warp
// (lane k of the half holds tile k; tiles beyond the vocabulary hold the
// identity (-inf, 0)).  M = max m_k; S = sum_k s_k exp(s (m_k - M)) summed as
// a fixed pairwise tree in tile-index order (issue #241 PR 3 merge formula).
// m_k - M is exact for 16-bit inputs; exp is the accurate library expf.  All
// 32 lanes call this together; every lane gets (M, S) of its half.
__device__ __forceinline__ MS tile_fold16(MS p, float s) {
    float M = p.m;
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off, 16));
    float term = (p.m == -INFINITY) ? 0.f : __fmul_rn(p.s, expf(__fmul_rn(s, __fsub_rn(p.m, M))));
#pragma unroll
    for (int off = 1; off <= 8; off <<= 1)
        term = __fadd_rn(term, __shfl_xor_sync(0xffffffffu, term, off, 16));
    return MS{M, term};
}

// LSE = s M + log S and logp = s x_y - LSE, carried in double (s M and s x_y
// are exact there) and each output rounded once to binary32 (the "downcast at
// final write" of issue #241 Goal).  lse_lo, when given, receives the binary32
// rounding residual of the LSE (LSE - lse), so that lse + lse_lo carries the
// LSE to about 2^-48 relative for the backward.
__device__ __forceinline__ void finalize_row(MS f, bool active, float x_y, float s, float* logp_out,
                                             float* lse_out, float* lse_lo_out) {
    const double l = (f.m == -INFINITY) ? -(double)INFINITY
                                        : (double)s * (double)f.m + log((double)f.s);
    const float lf = __double2float_rn(l);
    *lse_out = lf;
    if (lse_lo_out) *lse_lo_out = isfinite(lf) ? __double2float_rn(l - (double)lf) : 0.f;
    *logp_out = active ? __double2float_rn((double)s * (double)x_y - l) : 0.f;
}

__device__ __forceinline__ bool row_active(const uint8_t* mask, int64_t t, int64_t y, int64_t v,
                                           int64_t ignore_index) {
    return (mask == nullptr || __ldg(mask + t) != 0) && y >= 0 && y < v && y != ignore_index;
}

// ---------------------------------------------------------------- forward kernels

// Forward with plain loads (any alignment): one CTA of 16 warps per row, warp
// k reduces tile k.
template <Dt D, bool kScaled>
__global__ void __launch_bounds__(kFwdThreads)
k_logp_fwd(const void* __restrict__ x, int64_t n, int64_t v, int64_t ld, int64_t W,
           const int64_t* __restrict__ y, int64_t ignore_index, const uint8_t* __restrict__ mask,
           Scale sc, float* __restrict__ logp, float* __restrict__ lse, float* __restrict__ lse_lo) {
    __shared__ float sh_m[kTiles], sh_s[kTiles];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int EB = Unit<D>::kElemBytes;
    for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
        const char* xr = reinterpret_cast<const char*>(x) + t * ld * EB;
        bool act = false;
        float x_y = 0.f;
        if (threadIdx.x == 0) {
            const int64_t yt = __ldg(y + t);
            act = row_active(mask, t, yt, v, ignore_index);
            if (act) x_y = elem_value<D>(xr, yt);
        }
        const int64_t c0 = (int64_t)warp * W;
        const int64_t width = c0 >= v ? 0 : (v - c0 < W ? v - c0 : W);
        const MS p = tile_partial<kScaled>(tile_scan<D, false, kScaled>(xr + c0 * EB, width, lane, sc), sc);
        if (lane == 0) {
            sh_m[warp] = p.m;
            sh_s[warp] = p.s;
        }
        __syncthreads();
        if (warp == 0) {
            const int k = lane & 15;
            const MS f = tile_fold16(MS{sh_m[k], sh_s[k]}, sc.s);
            if (lane == 0)
                finalize_row(f, act, x_y, sc.s, logp + t, lse + t, lse_lo ? lse_lo + t : nullptr);
        }
        __syncthreads();
    }
}

// Forward with bulk copies (16-byte aligned rows whose byte stride is a
// multiple of 16, V < 2^31).  Persistent CTAs of 16 warps; CTA b takes rows
// b, b + grid, b + 2 grid, ...  Each warp streams its tile of successive rows
// through a private ring of kStages shared-memory stages (one group of 128
// units each): lane 0 issues cp.async.bulk for group i + kStages as soon as the
// warp has read group i, so copies of the next row are already in flight while
// a row is finished.  The lanes read the same words, in the same order, as
// tile_scan would load them (a ragged last unit is read from global memory),
// so results are bitwise those of k_logp_fwd.  Tile partials go to a
// double-buffered shared array; after one barrier per row, warp (row mod 16)
// merges them and writes the row.  A wait that runs out sets g_device_error;
// the warp then stops issuing copies and skips waits, and drains its copies in
// flight before exiting.
template <Dt D, bool kScaled>
__global__ void __launch_bounds__(kFwdThreads, kFwdMinBlocks<D>)
k_logp_fwd_bulk(const void* __restrict__ x, int64_t n, int64_t v, int64_t ld, int64_t W,
                const int64_t* __restrict__ y, int64_t ignore_index, const uint8_t* __restrict__ mask,
                Scale sc, float* __restrict__ logp, float* __restrict__ lse,
                float* __restrict__ lse_lo) {
    constexpr int EB = Unit<D>::kElemBytes;
    constexpr int UB = Unit<D>::kBytes;
    constexpr int SB = kStageBytes<D>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float sh_m[2][kTiles], sh_s[2][kTiles];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t stage0 = smem_u32(smem + warp * kStages * SB);
    const uint32_t bar0 = smem_u32(smem + kTiles * kStages * SB) + warp * kStages * 8;
    if (threadIdx.x < kTiles * kStages) mbar_init(smem_u32(smem + kTiles * kStages * SB) + threadIdx.x * 8, 1);
    fence_mbar_init();
    __syncthreads();

    // tile-local extents fit in 32 bits (the host routes V >= 2^31 elsewhere)
    const int64_t c0 = (int64_t)warp * W;
    const int width = (int)(c0 >= v ? 0 : (v - c0 < W ? v - c0 : W));
    const int nfull = width >> 3, nunit = (width + 7) >> 3;
    const int G = (nunit + kGroupUnits - 1) / kGroupUnits;       // groups per row
    const int Gfull = nfull / kGroupUnits;                       // groups of 128 full units
    const int64_t rows = (n > (int64_t)blockIdx.x) ? (n - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t jobs = rows * G;
    const int64_t row_step = (int64_t)gridDim.x * ld * EB;      // bytes

    // Issuer: group iss_g of the row at iss_row (its first byte of this tile),
    // stage iss_st.  Every lane tracks it; lane 0 issues.
    const char* iss_row = reinterpret_cast<const char*>(x) + ((int64_t)blockIdx.x * ld + c0) * EB;
    int iss_g = 0, iss_st = 0;
    int64_t issued = 0;
    auto issue_next = [&]() {
        if (lane == 0) {
            const int nv = nfull - iss_g * kGroupUnits;
            const uint32_t bytes = nv <= 0 ? 0u : (uint32_t)((nv < kGroupUnits ? nv : kGroupUnits) * UB);
            const uint32_t bar = bar0 + iss_st * 8;
            mbar_arrive_expect_tx(bar, bytes);
            if (bytes) bulk_g2s(stage0 + iss_st * SB, iss_row + (int64_t)iss_g * SB, bytes, bar);
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
        const char* xr = reinterpret_cast<const char*>(x) + t * ld * EB;
        bool act = false;
        float x_y = 0.f;
        if (warp == folder && lane == 0) {
            const int64_t yt = __ldg(y + t);
            act = row_active(mask, t, yt, v, ignore_index);
            if (act) x_y = elem_value<D>(xr, yt);
        }
        const char* tile = xr + c0 * EB;
        float m = -INFINITY, s = 0.f;
        for (int g = 0; g < G; ++g) {
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar0 + st * 8, phase, kWaitLimitCycles));
                if (!ok) fail_at = j * G + g;
            }
            const uint32_t sbase = stage0 + st * SB + lane * UB;
            Unit<D> q[kGroup];
            if (g < Gfull) {
#pragma unroll
                for (int u = 0; u < kGroup; ++u) unit_load_shared<D>(sbase + u * (kWarp * UB), q[u]);
                __syncwarp();
                if (ok && issued < jobs) {
                    if (lane == 0) fence_proxy_async_smem();
                    issue_next();
                }
                group_update<D, true, kScaled>(q, kGroup, m, s, sc);
            } else {
                const int v0 = g * kGroupUnits;
                int nvalid = 0;
#pragma unroll
                for (int u = 0; u < kGroup; ++u) {
                    const int jv = v0 + kWarp * u + lane;
                    if (jv < nfull) {
                        unit_load_shared<D>(sbase + u * (kWarp * UB), q[u]);
                        nvalid = u + 1;
                    } else if (jv < nunit) {
                        unit_load<D, false>(tile, (int64_t)jv * 8, width, q[u]);
                        nvalid = u + 1;
                    } else {
                        unit_fill_neg_inf<D>(q[u]);
                    }
                }
                __syncwarp();
                if (ok && issued < jobs) {
                    if (lane == 0) fence_proxy_async_smem();
                    issue_next();
                }
                if (nvalid == kGroup) group_update<D, true, kScaled>(q, nvalid, m, s, sc);
                else group_update<D, false, kScaled>(q, nvalid, m, s, sc);
            }
            if (++st == kStages) {
                st = 0;
                phase ^= 1u;
            }
        }
        const MS p = tile_partial<kScaled>(MS{m, s}, sc);
        if (lane == 0) {
            sh_m[j & 1][warp] = p.m;
            sh_s[j & 1][warp] = p.s;
        }
        __syncthreads();
        if (warp == folder) {
            const int k = lane & 15;
            const MS f = tile_fold16(MS{sh_m[j & 1][k], sh_s[j & 1][k]}, sc.s);
            if (lane == 0)
                finalize_row(f, act, x_y, sc.s, logp + t, lse + t, lse_lo ? lse_lo + t : nullptr);
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
template <Dt D, bool kVec, bool kScaled>
__global__ void __launch_bounds__(kFwdThreads)
k_logp_partials(const void* __restrict__ xs, int64_t n, int64_t ld, int64_t real_width, int64_t W,
                int tile0, int64_t vocab_start, const int64_t* __restrict__ y, Scale sc,
                float* __restrict__ pm, float* __restrict__ ps, float* __restrict__ sel) {
    constexpr int EB = Unit<D>::kElemBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
        const char* xr = reinterpret_cast<const char*>(xs) + t * ld * EB;
        if (threadIdx.x == 0) {
            const int64_t yt = __ldg(y + t);
            if (yt >= vocab_start && yt < vocab_start + real_width)
                sel[t] = elem_value<D>(xr, yt - vocab_start);
        }
        const int64_t c0 = (int64_t)warp * W;
        const int64_t width = real_width - c0 < W ? real_width - c0 : W;
        const MS p = tile_partial<kScaled>(tile_scan<D, kVec, kScaled>(xr + c0 * EB, width, lane, sc), sc);
        if (lane == 0) {
            pm[t * kTiles + tile0 + warp] = p.m;
            ps[t * kTiles + tile0 + warp] = p.s;
        }
    }
}

// Merge of tile partials: one half warp per row, the same tile_fold16 and
// finalize_row as the forward.  The partials may come from several ranks of
// a vocabulary-parallel group, gathered side by side: rank r's [n, 16] maxima,
// [n, 16] sums and [n] selected logits start rank_stride floats after rank
// r - 1's, and tile k is read from rank (tile_rank >> 4k) & 15, the rank that
// reduced it; the selected logit of row t from the rank owning the tile of
// its target, y_t / W.  On one GPU (all shards writing one buffer) the stride
// and the table are 0.  Only transport differs, so the bits are the same.
__global__ void __launch_bounds__(256)
k_logp_merge(const float* __restrict__ pm, const float* __restrict__ ps,
             const float* __restrict__ sel, const int64_t* __restrict__ y, int64_t ignore_index,
             const uint8_t* __restrict__ mask, int64_t n, int64_t v, int n_tiles, float s,
             float* __restrict__ logp, float* __restrict__ lse, float* __restrict__ lse_lo,
             int64_t rank_stride, uint64_t tile_rank, int64_t W) {
    const int lane = threadIdx.x & 31, k = lane & 15;
    const int64_t warp_g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t my_off = (int64_t)((tile_rank >> (4 * k)) & 15u) * rank_stride;
    for (int64_t pair = warp_g; 2 * pair < n; pair += n_warps) {
        const int64_t t = 2 * pair + (lane >> 4);
        const bool valid = t < n;
        MS p{-INFINITY, 0.f};
        if (valid && k < n_tiles) {
            p.m = __ldg(pm + my_off + t * kTiles + k);
            p.s = __ldg(ps + my_off + t * kTiles + k);
        }
        const MS f = tile_fold16(p, s);
        if (valid && k == 0) {
            const int64_t yt = __ldg(y + t);
            const bool act = row_active(mask, t, yt, v, ignore_index);
            const int64_t owner = act ? (int64_t)((tile_rank >> (4 * (int)(yt / W))) & 15u) : 0;
            const float x_y = act ? __ldg(sel + owner * rank_stride + t) : 0.f;
            finalize_row(f, act, x_y, s, logp + t, lse + t, lse_lo ? lse_lo + t : nullptr);
        }
    }
}

// ---------------------------------------------------------------- backward

// Per-row constants of the backward (see k_logp_bwd).
struct BwdRow {
    u64 neg_lr;        // (-lse_r, -lse_r)
    u64 s2;            // (s, s)
    u64 coef2;         // (coef, coef), coef = -s g (1 - delta)
    uint32_t floor_w;  // BF16: packed floor for the raw logits
    float floor_f;     // FP16/FP32: floor for the raw logits
    float lr, delta, gs, s;
};

// The pair (x_{2k}, x_{2k+1}) of a unit widened to binary32 and raised to the
// row's floor.
template <Dt D>
__device__ __forceinline__ u64 bwd_pair(const Unit<D>& u, int k, const BwdRow& r) {
    if constexpr (D == Dt::BF16) {
        const uint32_t w = bf2_max(u.w[k], r.floor_w);
        return f2(bf_lo(w), bf_hi(w));
    } else if constexpr (D == Dt::F16) {
        return f2(fmaxf(h_lo(u.w[k]), r.floor_f), fmaxf(h_hi(u.w[k]), r.floor_f));
    } else {
        return f2(fmaxf(__uint_as_float(u.w[2 * k]), r.floor_f),
                  fmaxf(__uint_as_float(u.w[2 * k + 1]), r.floor_f));
    }
}

// Output word(s) of a gradient pair in dtype D (for FP32 two words).
template <Dt D>
__device__ __forceinline__ void put_pair(uint32_t (&o)[Unit<D>::kWords], int k, float d0, float d1) {
    if constexpr (D == Dt::BF16) o[k] = pack_bf16x2(d0, d1);
    else if constexpr (D == Dt::F16) o[k] = pack_f16x2(d0, d1);
    else {
        o[2 * k] = __float_as_uint(d0);
        o[2 * k + 1] = __float_as_uint(d1);
    }
}

// Gradient of one unit (8 columns) into output words o, target column jt (or
// outside [0, 8)).
template <Dt D>
__device__ __forceinline__ void bwd_unit(const Unit<D>& u, const BwdRow& r, int64_t jt,
                                         uint32_t (&o)[Unit<D>::kWords]) {
    const u64 l2e = f2(kLog2e, kLog2e);
    const u64 nln2hi = f2(-kLn2Hi, -kLn2Hi), nln2lo = f2(-kLn2Lo, -kLn2Lo);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const u64 tt = f2_fma(bwd_pair<D>(u, k, r), r.s2, r.neg_lr);
        const u64 a = f2_mul(tt, l2e);
        const u64 c = f2_fma(a, nln2lo, f2_fma(a, nln2hi, tt));
        float a0, a1;
        f2_split(a, a0, a1);
        const u64 q = f2_mul(f2(ex2_ftz(a0), ex2_ftz(a1)), r.coef2);
        float d0, d1;
        f2_split(f2_fma(q, c, q), d0, d1);
        put_pair<D>(o, k, d0, d1);
    }
    if (jt >= 0 && jt < 8) {
        // target column: s g (1 - p) without cancellation, patched into its word
        // (the element is picked by unrolled selects: no run-time index)
        const int kt = (int)(jt >> 1);
        float xt = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float lo, hi;
            f2_split(bwd_pair<D>(u, k, r), lo, hi);
            if (k == kt) xt = (jt & 1) ? hi : lo;
        }
        const float dt = __fmul_rn(-r.gs, expm1f(__fsub_rn(__fmaf_rn(r.s, xt, -r.lr), r.delta)));
        if constexpr (D == Dt::F32) {
            // blend by masks (a predicated store per word would be folded into
            // one store at a run-time index, which needs local memory)
            const uint32_t bits = __float_as_uint(dt);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t msk = 0u - (uint32_t)(j == (int)jt);
                o[j] = (o[j] & ~msk) | (bits & msk);
            }
        } else {
            const uint32_t bt = ((D == Dt::BF16) ? pack_bf16x2(dt, dt) : pack_f16x2(dt, dt)) & 0xffffu;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (k == kt) o[k] = (jt & 1) ? ((o[k] & 0xffffu) | (bt << 16)) : ((o[k] & 0xffff0000u) | bt);
        }
    }
}

template <Dt D, bool kVecIn, bool kInPlace>
__device__ __forceinline__ void bwd_load(const char* xr, int64_t col, int64_t v, Unit<D>& u) {
    constexpr int EB = Unit<D>::kElemBytes;
    if (kVecIn && col + 8 <= v) {
        const char* p = xr + col * EB;
        const uint4 a = kInPlace ? ld_v4(p) : ld_nc_v4(p);
        u.w[0] = a.x; u.w[1] = a.y; u.w[2] = a.z; u.w[3] = a.w;
        if constexpr (D == Dt::F32) {
            const uint4 b = kInPlace ? ld_v4(p + 16) : ld_nc_v4(p + 16);
            u.w[4] = b.x; u.w[5] = b.y; u.w[6] = b.z; u.w[7] = b.w;
        }
    } else if constexpr (D == Dt::F32) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            u.w[j] = (col + j < v) ? (kInPlace ? elem_bits_plain<D>(xr, col + j) : elem_bits<D>(xr, col + j)) : 0u;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t lo = 0, hi = 0;
            if (col + 2 * k < v)
                lo = kInPlace ? elem_bits_plain<D>(xr, col + 2 * k) : elem_bits<D>(xr, col + 2 * k);
            if (col + 2 * k + 1 < v)
                hi = kInPlace ? elem_bits_plain<D>(xr, col + 2 * k + 1) : elem_bits<D>(xr, col + 2 * k + 1);
            u.w[k] = lo | (hi << 16);
        }
    }
}

template <Dt D, bool kVecOut>
__device__ __forceinline__ void bwd_store(char* dr, int64_t col, int64_t v,
                                          const uint32_t (&o)[Unit<D>::kWords]) {
    constexpr int EB = Unit<D>::kElemBytes;
    if (kVecOut && col + 8 <= v) {
        st_cs_v4(dr + col * EB, make_uint4(o[0], o[1], o[2], o[3]));
        if constexpr (D == Dt::F32) st_cs_v4(dr + col * EB + 16, make_uint4(o[4], o[5], o[6], o[7]));
    } else if constexpr (D == Dt::F32) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (col + j < v) reinterpret_cast<uint32_t*>(dr)[col + j] = o[j];
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (col + j < v)
                reinterpret_cast<uint16_t*>(dr)[col + j] =
                    (uint16_t)((j & 1) ? (o[j >> 1] >> 16) : (o[j >> 1] & 0xffffu));
    }
}

// Backward: one CTA per (segment of kBwdSegCols columns, row), elementwise.
// Per active row: LSE = lse (+ lse_lo) is split as lse_r + delta with lse_r
// on a 2^-16 grid, so that t = s x - lse_r is exact for the bulk of BF16
// logits at s = 1 (one rounding otherwise); exp(t) = 2^a (1 + c) with
// a = t log2 e rounded and c = t - a ln 2 recovered by two fused multiply-adds
// against a two-float ln 2 (the rounding error of a, carried to first order);
// coef = -s g (1 - delta) ~ -s g exp(-delta) folds s, g and delta in once per
// row, with the exp2 bias correction.  Logits below about (LSE - 200) / s are raised to that bound first (their
// exp is below e^-199, zero in binary32), which also keeps a -inf logit from
// producing inf - inf.  The target column is s g (1 - p) = -s g expm1(s x - LSE),
// without cancellation.  Values below 2^-126 flush to zero.  Each thread loads
// its eight units before computing any, so eight (FP32: sixteen) 16-byte loads
// are in flight per thread.
//
// Vocabulary shards: the buffer holds global columns [y_off, y_off + v) of a
// v_total-column vocabulary (unsharded: y_off = 0, v_total = v).  A row is
// active by its global target (in [0, v_total)); the one-hot term lands on
// local column y_t - y_off only when that lies in [0, v).  Every element is
// computed from the same per-row constants as in the unsharded call, so the
// shards' outputs side by side are the unsharded gradient bit for bit.
template <Dt D, bool kVecIn, bool kVecOut, bool kInPlace>
__global__ void __launch_bounds__(kBwdThreads, kBwdMinBlocks<D>)
k_logp_bwd(const void* x, int64_t n, int64_t v, int64_t ld, const int64_t* __restrict__ y,
           int64_t ignore_index, const uint8_t* __restrict__ mask, float s, float inv_s,
           const float* __restrict__ lse, const float* __restrict__ lse_lo,
           const float* __restrict__ g, void* dx, int64_t ld_out, int64_t y_off, int64_t v_total) {
    constexpr int EB = Unit<D>::kElemBytes;
    constexpr int NW = Unit<D>::kWords;
    // grid: x = segment of the row, y = row (strided when n > gridDim.y)
    const int64_t col0 = (int64_t)blockIdx.x * kBwdSegCols + (int64_t)threadIdx.x * 8;
#pragma unroll 1
    for (int64_t t = blockIdx.y; t < n; t += gridDim.y) {
        const char* xr = reinterpret_cast<const char*>(x) + t * ld * EB;
        char* dr = reinterpret_cast<char*>(dx) + t * ld_out * EB;
        const int64_t yt = __ldg(y + t);
        const int64_t cs = (int64_t)kBwdThreads * 8;
        if (!row_active(mask, t, yt, v_total, ignore_index)) {
            uint32_t z[NW];
#pragma unroll
            for (int k = 0; k < NW; ++k) z[k] = 0u;
#pragma unroll
            for (int u = 0; u < kBwdUnitsPerThread; ++u)
                if (col0 + u * cs < v) bwd_store<D, kVecOut>(dr, col0 + u * cs, v, z);
            continue;
        }
        BwdRow r;
        const float l = __ldg(lse + t);
        const float l_lo = lse_lo ? __ldg(lse_lo + t) : 0.f;
        r.s = s;
        r.gs = __fmul_rn(s, __ldg(g + t));
        r.lr = (fabsf(l) < 8388608.f) ? __fmul_rn(rintf(__fmul_rn(l, 65536.f)), 1.f / 65536.f) : l;
        r.delta = __fadd_rn(__fsub_rn(l, r.lr), l_lo);           // l - lr is exact
        // -s g (1 - delta), times (1 + b) for the mean bias b of ex2.approx
        const float coef = __fmaf_rn(r.gs, __fsub_rn(r.delta, kEx2BiasComp), -r.gs);
        const float fl = __fmul_rn(__fsub_rn(l, 200.f), inv_s);   // ~ (LSE - 200) / s
        r.floor_f = fl;
        r.floor_w = 0xff80ff80u;
        if constexpr (D == Dt::BF16) {
            const uint32_t b = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rd(fl));
            r.floor_w = b | (b << 16);
        }
        r.neg_lr = f2(-r.lr, -r.lr);
        r.s2 = f2(s, s);
        r.coef2 = f2(coef, coef);

        Unit<D> w[kBwdUnitsPerThread];
#pragma unroll
        for (int u = 0; u < kBwdUnitsPerThread; ++u)
            if (col0 + u * cs < v) bwd_load<D, kVecIn, kInPlace>(xr, col0 + u * cs, v, w[u]);
#pragma unroll
        for (int u = 0; u < kBwdUnitsPerThread; ++u) {
            if (col0 + u * cs < v) {
                uint32_t o[NW];
                bwd_unit<D>(w[u], r, yt - y_off - (col0 + u * cs), o);
                bwd_store<D, kVecOut>(dr, col0 + u * cs, v, o);
            }
        }
    }
}

// Mean relative error of ex2.approx.ftz.f32 against the double exp2 over a
// fixed grid of 2^20 arguments in [-24, 0) (one CTA; fixed reduction order).
__device__ double g_ex2_bias;
__global__ void __launch_bounds__(1024) k_ex2_bias_selftest() {
    __shared__ double sh[32];
    double acc = 0.0;
    for (int i = threadIdx.x; i < (1 << 20); i += 1024) {
        const float a = -24.0f * (float)i / (float)(1 << 20) - 1.0e-6f * (float)(i & 1023);
        const double ref = exp2((double)a);
        acc += ((double)ex2_ftz(a) - ref) / ref;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < 32; ++w) t += sh[w];
        g_ex2_bias = t / (double)(1 << 20);
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
