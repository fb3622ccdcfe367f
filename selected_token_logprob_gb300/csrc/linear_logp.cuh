// Fused LM head + selected-token log-probability on the fifth-generation
// tensor cores (tcgen05) of sm_103a.
//
// linear_logp is named in RL-Kernel PR #495 (Summary) and nowhere specified;
// here it is the selected-token logprob of issue #241 (Background, Goal)
// taken of s z, where z = H W^T are the logits of BF16 hidden states
// H [N, D] against BF16 LM-head weight rows W [V, D].  The logits never reach
// memory: each 128 x 256 tile of z is accumulated in tensor memory and reduced
// there to per-row (max, sumexp) tile partials, which a second kernel merges
// in fixed tile order (the partials-and-merge structure of issue #241 PR 3).
//
// Contraction kernel, one persistent CTA per SM, 6 warps:
//   warp 0      TMA producer: for each tile and each 64-wide K block, one
//               tensor-map copy of the H block (128 x 64) and one of the W
//               block (256 x 64) into a 4-stage shared-memory ring (192 KB in
//               flight: the L2 latency under load is what the ring covers),
//               both with 128-byte swizzle, completing on the stage's mbarrier
//               (64-byte swizzle with 32-wide K blocks and 9 stages measured
//               slower: the tensor pipe reads those operands more slowly);
//   warp 1      allocates 512 TMEM columns (two 128 x 256 FP32 accumulators),
//               and one elected lane issues tcgen05.mma (kind::f16, BF16 in,
//               FP32 accumulate, M = 128, N = 256, K = 16), four per K block,
//               committing each stage back to the producer and each finished
//               accumulator to the epilogue;
//   warps 2-5   epilogue: warp w reads TMEM lanes 32 (w mod 4) .. +31, one
//               row per thread, 32 columns at a time, and forms the row's
//               tile partial (m = max z over the tile's real columns,
//               s = sum exp(s (z - m)) with the exponent to full binary32
//               accuracy) and, in the tile that holds the row's target, the
//               selected logit; the accumulator is released as soon as it is
//               read, so the epilogue of tile i overlaps the MMAs of tile i+1.
// Tiles are visited in groups of 32 row blocks (vocabulary tiles outer, row
// blocks inner) so that the CTAs running at one time share their W and H
// blocks in L2 and the weight is read from DRAM once per group (a sweep of 16
// to 64 measured 32 and 48 fastest; 64 thrashes L2).  A row's partials do not depend on which CTA, in which order,
// computed them: each logit is one tensor-core dot product over K in a fixed
// order, so the result is batch-invariant and deterministic.
//
// Every wait is bounded: a wait that runs out sets the sticky device error
// word and a CTA-wide abort flag; every role then stops, the producer waits
// (bounded) for its copies in flight, the MMA lane for its MMAs, and TMEM is
// freed before the CTA exits.
#pragma once

#include <cuda.h>

#include "logp_kernels.cuh"

namespace flp {

constexpr int kLinBM = 128;                 // rows (tokens) per tile: UMMA M
constexpr int kLinBN = 256;                 // vocabulary columns per tile: UMMA N
constexpr int kLinBK = 64;                  // K per stage: one 128-byte swizzle row of BF16
constexpr int kLinUmmaK = 16;               // K of one tcgen05.mma kind::f16
constexpr int kLinStages = 4;               // 4 x 48 KB in flight per SM
constexpr int kLinThreads = 192;            // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kLinGroupRows = 32;           // row blocks per raster group (swept: 16-64)
constexpr uint32_t kLinABytes = kLinBM * kLinBK * 2;
constexpr uint32_t kLinBBytes = kLinBN * kLinBK * 2;
constexpr uint32_t kLinStageBytes = kLinABytes + kLinBBytes;
constexpr uint32_t kLinTmemCols = 2 * kLinBN;   // two accumulators
constexpr uint32_t kLinBarBytes = 256;
constexpr size_t kLinSmemBytes = 1024 + (size_t)kLinStages * kLinStageBytes + kLinBarBytes;
// Swizzle of the staged operands: the K extent of a stage row, in bytes (64:
// 64-byte swizzle, 128: 128-byte swizzle), and its 8-row repeat.
constexpr uint32_t kLinRowBytes = kLinBK * 2;
constexpr uint32_t kLinAtomBytes = 8 * kLinRowBytes;
static_assert(kLinRowBytes == 64 || kLinRowBytes == 128, "stage rows must be one swizzle span");
static_assert(kLinSmemBytes <= 232448, "shared memory per CTA");
static_assert(2 * kLinStages * 8 + 48 <= kLinBarBytes, "barrier block");
constexpr int kLinMergeThreads = 256;

// Instruction descriptor of tcgen05.mma kind::f16: D in FP32 (bits 4-5 = 1),
// A and B in BF16 (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16
// = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kLinIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                               ((uint32_t)(kLinBN >> 3) << 17) | ((uint32_t)(kLinBM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand stored as rows of
// kLinRowBytes with the matching swizzle (the layout the tensor-map copy
// writes): start address >> 4 in bits 0-13, leading byte offset (unused for
// this layout; 16 B) in bits 16-29, stride byte offset = 8 rows in bits
// 32-45, the descriptor version 1 in bits 46-47, the swizzle mode in bits
// 61-63 (2: 128-byte, 4: 64-byte).  The buffer is 1024-byte aligned; the K
// step of 16 BF16 (32 B) inside the swizzle row advances the start address.
__device__ __forceinline__ uint64_t umma_desc_swz(uint32_t saddr) {
    constexpr uint64_t mode = (kLinRowBytes == 128) ? 2 : 4;
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(kLinAtomBytes >> 4) << 32) | ((uint64_t)1 << 46) | (mode << 61);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D (+)= A B^T for one K = 16 slice; accumulate = 0 overwrites D.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 32 consecutive binary32 columns of this thread's TMEM lane (shape 32x32b,
// 32 repetitions), waited for inside the same statement so that no use of the
// registers can be scheduled before the data is there.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Bounded wait on an mbarrier phase that also gives up once another role of
// the CTA has raised the abort flag.
__device__ __forceinline__ bool lin_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kWaitLimitCycles) {
                *abort_flag = 1;
                atomicExch(&g_device_error, 1);
                return false;
            }
        }
    }
}

struct LinTile {
    int rb, vt;
};

// Tile i of the raster: groups of kLinGroupRows row blocks; inside a group
// the vocabulary tile is the slow index and the row block the fast one.
__device__ __forceinline__ LinTile lin_tile(int64_t i, int nrb, int nvt) {
    const int64_t per_group = (int64_t)kLinGroupRows * nvt;
    const int g = (int)(i / per_group);
    const int r = (int)(i - (int64_t)g * per_group);
    const int rows = min(kLinGroupRows, nrb - g * kLinGroupRows);
    return LinTile{g * kLinGroupRows + r % rows, r / rows};
}

struct LinArgs {
    int64_t n, v;           // rows; vocabulary columns held by this call's weight rows
    int nrb, nvt, nkb;      // row blocks, vocabulary tiles of this call, K blocks
    // vocabulary sharding: this call's weight rows are global columns
    // [vocab_start, vocab_start + v) of a v_total-column vocabulary whose
    // partials are laid out [n, nvt_total]; this call's tiles are global tiles
    // [vt0, vt0 + nvt).  Unsharded: vocab_start = vt0 = 0, v_total = v.
    int64_t vocab_start, v_total;
    int vt0, nvt_total;
    const int64_t* y;
    int64_t ignore_index;
    const uint8_t* mask;
    Scale sc;
    float* pm;     // [n, nvt] tile maxima (row-major: a row's partials are contiguous)
    float* ps;     // [n, nvt] tile sums
    float* xsel;   // [n] selected logit z[t, y_t] (active rows)
    // gradient mode: rows [n_valid, n) are padding and get zero gradients
    int64_t n_valid;
    const float* lse;
    const float* lse_lo;   // nullable
    const float* g;
    float inv_s;
    uint16_t* dz;          // [n, ld_dz] BF16 dZ; columns [v, ld_dz) are written as 0
    int64_t ld_dz;
};

// Per-row constants of dZ = s g (onehot - exp(s z - LSE)), split like the
// logits backward: LSE (+ its residual) = lr + delta with lr on a 2^-16 grid,
// coef = -s g (1 - delta + b) with b the mean exp2 bias, and logits below
// (LSE - 200) / s raised to that bound (their exp is 0 in binary32).
struct LinGradRow {
    float s, lr, delta, gs, coef, floor_f;
};

__device__ __forceinline__ LinGradRow lin_grad_row(float l, float l_lo, float g, float s, float inv_s) {
    LinGradRow r;
    r.s = s;
    r.gs = __fmul_rn(s, g);
    r.lr = (fabsf(l) < 8388608.f) ? __fmul_rn(rintf(__fmul_rn(l, 65536.f)), 1.f / 65536.f) : l;
    r.delta = __fadd_rn(__fsub_rn(l, r.lr), l_lo);                // l - lr is exact
    r.coef = __fmaf_rn(r.gs, __fsub_rn(r.delta, kEx2BiasComp), -r.gs);
    r.floor_f = __fmul_rn(__fsub_rn(l, 200.f), inv_s);
    return r;
}

// dZ of one 32-column chunk of a row as 16 BF16 pairs: exp(t) = 2^a (1 + c)
// with t = s z - lr, a = t log2 e rounded, c = t - a ln 2 by two fused
// multiply-adds against a two-float ln 2; the target column jt (if in
// [0, 32)) as -s g expm1(s z - LSE); columns at or beyond nvalid are 0.
__device__ __forceinline__ void lin_grad_chunk(const uint32_t (&r)[32], const LinGradRow& g, int jt, int nvalid,
                                               uint32_t (&o)[16]) {
    float d[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float z = fmaxf(__uint_as_float(r[j]), g.floor_f);
        const float t = __fmaf_rn(z, g.s, -g.lr);
        const float a = __fmul_rn(t, kLog2e);
        const float c = __fmaf_rn(a, -kLn2Lo, __fmaf_rn(a, -kLn2Hi, t));
        const float q = __fmul_rn(ex2_ftz(a), g.coef);
        d[j] = (j < nvalid) ? __fmaf_rn(q, c, q) : 0.f;
    }
    if (jt >= 0 && jt < 32) {
        float zt = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j == jt) zt = __uint_as_float(r[j]);
        const float dt = __fmul_rn(-g.gs, expm1f(__fsub_rn(__fmaf_rn(g.s, zt, -g.lr), g.delta)));
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j == jt) d[j] = dt;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = pack_bf16x2(d[2 * k], d[2 * k + 1]);
}

// Reduce one 32-column chunk of a row into (m, s): columns at or beyond
// `nvalid` are not part of the vocabulary.
__device__ __forceinline__ void lin_chunk(const uint32_t (&r)[32], int nvalid, const Scale& sc, float& m,
                                          float& s) {
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = (j < nvalid) ? __uint_as_float(r[j]) : -INFINITY;
    float c[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) c[j] = fmaxf(x[2 * j], x[2 * j + 1]);
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) c[j] = fmaxf(c[j], c[j + w]);
    const float mn = fmaxf(m, c[0]);
    // rescale the running sum when the maximum grows (m = -inf: s is 0)
    if (mn > m) s = (m == -INFINITY) ? 0.f : __fmul_rn(s, ex2_ftz(to_log2_1<true>(__fsub_rn(m, mn), sc)));
    m = mn;
    float e[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float a0 = to_log2_1<true>(__fsub_rn(x[2 * j], mn), sc);
        const float a1 = to_log2_1<true>(__fsub_rn(x[2 * j + 1], mn), sc);
        e[j] = __fadd_rn(ex2_ftz(a0), ex2_ftz(a1));
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) e[j] = __fadd_rn(e[j], e[j + w]);
    s = __fadd_rn(s, e[0]);
}

// kGrad = false: tile partials of the forward.  kGrad = true: the same
// contraction with an epilogue that writes dZ in BF16 (the backward's
// recomputation of the logits, which never reach memory in FP32).
template <bool kGrad>
__global__ void __launch_bounds__(kLinThreads, 1)
k_linear_logp_tiles(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                    LinArgs p) {
    extern __shared__ __align__(1024) unsigned char lin_smem_raw[];
    const uint32_t raw = smem_u32(lin_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + kLinStages * kLinStageBytes;
    // barrier block: full[4], empty[4], tfull[2], tempty[2], drain, tmem slot, abort flag
    const uint32_t full0 = bars, empty0 = bars + 8 * kLinStages;
    const uint32_t tfull0 = bars + 16 * kLinStages, tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    const uint32_t slot = drain + 8;
    unsigned char* slot_gen = lin_smem_raw + (slot - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(slot_gen);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slot_gen + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (int64_t)p.nrb * p.nvt;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLinStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_h);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc(slot, kLinTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int64_t i = blockIdx.x; ok && i < ntiles; i += gridDim.x) {
                const LinTile tl = lin_tile(i, p.nrb, p.nvt);
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!lin_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_dst = base + stage * kLinStageBytes;
                    mbar_arrive_expect_tx(full0 + 8 * stage, kLinStageBytes);
                    tma_load_2d(a_dst, &tm_h, kb * kLinBK, tl.rb * kLinBM, full0 + 8 * stage);
                    tma_load_2d(a_dst + kLinABytes, &tm_w, kb * kLinBK, tl.vt * kLinBN, full0 + 8 * stage);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == kLinStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // wait (bounded) for the copies this thread still has in flight
                for (int s = 0; s < kLinStages; ++s)
                    if (issued & (1u << s))
                        mbar_wait(full0 + 8 * s, (last_par >> s) & 1u, kWaitLimitCycles);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t i = blockIdx.x; ok && i < ntiles; i += gridDim.x) {
                if (!lin_wait(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * kLinBN);
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!lin_wait(full0 + 8 * stage, phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = base + stage * kLinStageBytes;
                    const uint64_t a_desc = umma_desc_swz(a_addr);
                    const uint64_t b_desc = umma_desc_swz(a_addr + kLinABytes);
#pragma unroll
                    for (int k = 0; k < kLinBK / kLinUmmaK; ++k) {
                        // K step of 16 BF16 = 32 bytes = 2 units of the 16-byte address field
                        umma_bf16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, kLinIdesc, (kb | k) != 0);
                    }
                    umma_commit(empty0 + 8 * stage);
                    if (++stage == kLinStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(tfull0 + 8 * acc);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA issued has completed before TMEM and shared memory go away
            umma_commit(drain);
            mbar_wait(drain, 0, kWaitLimitCycles);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: one row per thread
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t i = blockIdx.x; i < ntiles; i += gridDim.x) {
            const LinTile tl = lin_tile(i, p.nrb, p.nvt);
            if (!lin_wait(tfull0 + 8 * acc, acc_phase, abort_flag)) break;
            tc_fence_after();
            const int64_t t = (int64_t)tl.rb * kLinBM + row;
            const int64_t col0 = (int64_t)tl.vt * kLinBN;
            if constexpr (kGrad) {
                bool act = false;
                int64_t jt = -1;
                LinGradRow gr{};
                if (t < p.n_valid) {
                    const int64_t yt = __ldg(p.y + t);
                    act = row_active(p.mask, t, yt, p.v_total, p.ignore_index);
                    if (act) {
                        gr = lin_grad_row(__ldg(p.lse + t), p.lse_lo ? __ldg(p.lse_lo + t) : 0.f, __ldg(p.g + t),
                                          p.sc.s, p.inv_s);
                        const int64_t yl = yt - p.vocab_start;   // target column in this call's rows
                        if (yl >= col0 && yl < col0 + kLinBN) jt = yl - col0;
                    }
                }
                const int nreal = (p.v - col0 < kLinBN) ? (int)(p.v - col0) : kLinBN;
                uint16_t* drow = p.dz + t * p.ld_dz;
#pragma unroll 1
                for (int c = 0; c < kLinBN / 32; ++c) {
                    const int64_t c0 = col0 + c * 32;
                    if (c0 >= p.ld_dz) break;  // uniform over the CTA
                    __syncwarp();
                    uint32_t r[32];
                    tmem_ld32(lane_addr + (uint32_t)(acc * kLinBN + c * 32), r);
                    uint32_t o[16];
                    if (act) {
                        lin_grad_chunk(r, gr, (int)(jt - c * 32), nreal - c * 32, o);
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = 0u;
                    }
                    if (t < p.n) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            if (c0 + 8 * q4 < p.ld_dz)
                                st_cs_v4(drow + c0 + 8 * q4, make_uint4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]));
                    }
                }
                tc_fence_before();
                mbar_arrive(tempty0 + 8 * acc);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                continue;
            }
            int64_t jt = -1;  // target column inside this tile, if the row is active
            if (t < p.n) {
                const int64_t yt = __ldg(p.y + t);
                const int64_t yl = yt - p.vocab_start;   // target column in this call's weight rows
                if (row_active(p.mask, t, yt, p.v_total, p.ignore_index) && yl >= col0 && yl < col0 + kLinBN)
                    jt = yl - col0;
            }
            const int nreal = (p.v - col0 < kLinBN) ? (int)(p.v - col0) : kLinBN;
            float m = -INFINITY, s = 0.f, xs = 0.f;
#pragma unroll 1
            for (int c = 0; c < kLinBN / 32; ++c) {
                if (c * 32 >= nreal) break;  // uniform over the CTA
                __syncwarp();
                uint32_t r[32];
                tmem_ld32(lane_addr + (uint32_t)(acc * kLinBN + c * 32), r);
                if (jt >= c * 32 && jt < c * 32 + 32) {
                    const int j = (int)jt - c * 32;
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        if (k == j) xs = __uint_as_float(r[k]);
                }
                lin_chunk(r, nreal - c * 32, p.sc, m, s);
            }
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            if (t < p.n) {
                p.pm[t * p.nvt_total + p.vt0 + tl.vt] = m;
                p.ps[t * p.nvt_total + p.vt0 + tl.vt] = __fmaf_rn(s, kEx2BiasComp, s);
                if (jt >= 0) p.xsel[t] = xs;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kLinTmemCols);
    }
}

// Merge of the nvt tile partials of each row, one warp per row (rows strided
// over the grid): lane j folds partials j, j + 32, ... in that order, then the
// lanes combine with a fixed xor butterfly — M = max_k m_k first, then
// S = sum_k s_k exp(s (m_k - M)) with the accurate expf — and lane 0 finishes
// LSE = s M + log S and logp = s z_y - LSE in double (finalize_row).  The
// order depends only on nvt, never on n or on the grid.
__global__ void __launch_bounds__(kLinMergeThreads)
k_linear_logp_merge(const float* __restrict__ pm, const float* __restrict__ ps, const float* __restrict__ xsel,
                    int64_t n, int nvt, int64_t v, const int64_t* __restrict__ y, int64_t ignore_index,
                    const uint8_t* __restrict__ mask, float s, float* __restrict__ logp, float* __restrict__ lse,
                    float* __restrict__ lse_lo) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < n; t += warps) {
        const float* rm = pm + t * nvt;
        const float* rs = ps + t * nvt;
        float M = -INFINITY;
        for (int k = lane; k < nvt; k += 32) M = fmaxf(M, __ldg(rm + k));
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float S = 0.f;
        if (M != -INFINITY) {
            for (int k = lane; k < nvt; k += 32) {
                const float mk = __ldg(rm + k);
                if (mk != -INFINITY) S = __fmaf_rn(__ldg(rs + k), expf(__fmul_rn(s, __fsub_rn(mk, M))), S);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) S = __fadd_rn(S, __shfl_xor_sync(0xffffffffu, S, off));
        if (lane == 0) {
            const int64_t yt = __ldg(y + t);
            const bool act = row_active(mask, t, yt, v, ignore_index);
            const float x_y = act ? __ldg(xsel + t) : 0.f;
            finalize_row(MS{M, S}, act, x_y, s, logp + t, lse + t, lse_lo ? lse_lo + t : nullptr);
        }
    }
}

// The ranks of a vocabulary-parallel LM head, in the order of their first
// tile: rank rank[j] holds tiles [t0[j], t1[j]) of the 256-column grid.
constexpr int kLinMaxRanks = 16;
struct LinRankTiles {
    int world;
    int t0[kLinMaxRanks], t1[kLinMaxRanks], rank[kLinMaxRanks];
};

// The merge of k_linear_logp_merge over the ranks' all-gathered workspaces
// (rank r's at gathered + r * stride, laid out as the one-buffer workspace):
// tile k is read from the rank that holds it, the selected logit from the
// rank that holds the target's tile.  Each lane visits the same tiles in the
// same order with the same arithmetic, so the result is the one-buffer
// merge's bit for bit.
__global__ void __launch_bounds__(kLinMergeThreads)
k_linear_logp_merge_gathered(const float* __restrict__ gathered, int64_t stride, LinRankTiles rt, int64_t n, int nvt,
                             int64_t v, const int64_t* __restrict__ y, int64_t ignore_index,
                             const uint8_t* __restrict__ mask, float s, float* __restrict__ logp,
                             float* __restrict__ lse, float* __restrict__ lse_lo) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t ps_off = (int64_t)nvt * n, sel_off = 2 * (int64_t)nvt * n;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < n; t += warps) {
        float M = -INFINITY;
        int j = 0;
        for (int k = lane; k < nvt; k += 32) {
            while (j + 1 < rt.world && k >= rt.t1[j]) ++j;
            M = fmaxf(M, __ldg(gathered + rt.rank[j] * stride + t * nvt + k));
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float S = 0.f;
        if (M != -INFINITY) {
            j = 0;
            for (int k = lane; k < nvt; k += 32) {
                while (j + 1 < rt.world && k >= rt.t1[j]) ++j;
                const float* blk = gathered + rt.rank[j] * stride;
                const float mk = __ldg(blk + t * nvt + k);
                if (mk != -INFINITY) S = __fmaf_rn(__ldg(blk + ps_off + t * nvt + k), expf(__fmul_rn(s, __fsub_rn(mk, M))), S);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) S = __fadd_rn(S, __shfl_xor_sync(0xffffffffu, S, off));
        if (lane == 0) {
            const int64_t yt = __ldg(y + t);
            const bool act = row_active(mask, t, yt, v, ignore_index);
            float x_y = 0.f;
            if (act) {
                const int tile = (int)(yt / kLinBN);
                int o = 0;
                while (o + 1 < rt.world && tile >= rt.t1[o]) ++o;
                x_y = __ldg(gathered + rt.rank[o] * stride + sel_off + t);
            }
            finalize_row(MS{M, S}, act, x_y, s, logp + t, lse + t, lse_lo ? lse_lo + t : nullptr);
        }
    }
}

// out = ((b_0 + b_1) + b_2) + ... of `world` [rows, cols] FP32 blocks at
// blocks + r * stride (row pitch cols), one rounding per addition, in rank
// order: the sum the one-GPU sharded backward forms when each later shard
// adds its term of dhidden.
__global__ void __launch_bounds__(256) k_sum_blocks_ordered(const float* __restrict__ blocks, int64_t stride,
                                                            int world, int64_t rows, int64_t cols,
                                                            float* __restrict__ out, int64_t ldo) {
    const int64_t total = rows * cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        float acc = __ldg(blocks + i);
        for (int k = 1; k < world; ++k) acc = __fadd_rn(acc, __ldg(blocks + (int64_t)k * stride + i));
        out[r * ldo + c] = acc;
    }
}

}  // namespace flp
