// Plain BF16 x BF16 -> FP32 contraction on the tcgen05 tensor cores, for the
// two products of the fused LM head's backward (the method's backward, RL-Kernel
// PR #495 Summary item 2, taken through the contraction z = H W^T):
//   dH = dZ W      C[M = rows, N = D],  K = V:   A = dZ (K-major),  B = W (MN-major)
//   dW = dZ^T H    C[M = V,    N = D],  K = rows: A = dZ^T (MN-major), B = H (MN-major)
// Both operands are read where they lie: an operand whose contiguous axis is
// M (or N) is staged "MN-major" (tensor-map boxes of 64 M/N elements by 64 K
// rows, 128-byte swizzle) and the MMA's instruction descriptor marks it
// transposed, so nothing is transposed in memory.
//
// One persistent CTA per SM, 6 warps, the roles of the fused LM-head kernel:
//   warp 0      TMA producer: per K block of 64, the A tile (128 x 64) and the
//               B tile (256 x 64) into a 4-stage ring (48 KB per stage);
//   warp 1      allocates 512 TMEM columns (two 128 x 256 FP32 accumulators);
//               one lane issues tcgen05.mma kind::f16 (M = 128, N = 256,
//               K = 16), four per K block, committing stages and accumulators;
//   warps 2-5   epilogue: one output row per thread (TMEM lane), 32 columns at
//               a time, written as FP32 (or added to C: one rounding per
//               element, C + acc), so the next tile's MMAs overlap it.
// Work units are (K split, M block, N block), N fastest, so the CTAs running
// together share their A tiles (and, for dW, the whole B) in L2.  A split s
// covers K blocks [s nkb / S, (s + 1) nkb / S) and writes its own partial
// C + s * split_stride; a separate fixed-order pass adds the splits.  The
// split count depends only on the shape, so every result is deterministic and
// the same for any batch (each element is one tensor-core dot product over K
// in increasing order per split).
//
// Every wait is bounded (lin_wait): on a timeout the CTA raises its abort
// flag, all roles stop, in-flight copies and MMAs are drained, TMEM is freed.
#pragma once

#include "linear_logp.cuh"

namespace flp {

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kGemmABytes = kGemmBM * kGemmBK * 2;     // 16 KB
constexpr uint32_t kGemmBBytes = kGemmBN * kGemmBK * 2;     // 32 KB
constexpr uint32_t kGemmStageBytes = kGemmABytes + kGemmBBytes;
constexpr uint32_t kGemmBoxBytes = 64 * kGemmBK * 2;        // one MN-major box: 64 MN x 64 K
constexpr size_t kGemmSmemBytes = 1024 + (size_t)kGemmStages * kGemmStageBytes + 256;
static_assert(kGemmSmemBytes <= 232448, "shared memory per CTA");

// Instruction descriptor (kind::f16): D FP32, A and B BF16, M = 128, N = 256,
// bit 15 = A MN-major, bit 16 = B MN-major.
template <bool kAmn, bool kBmn>
__host__ __device__ constexpr uint32_t gemm_idesc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((kAmn ? 1u : 0u) << 15) | ((kBmn ? 1u : 0u) << 16) |
           ((uint32_t)(kGemmBN >> 3) << 17) | ((uint32_t)(kGemmBM >> 4) << 24);
}

// Shared-memory descriptor of an MN-major operand with 128-byte swizzle, as
// the tensor-map boxes lay it out: each K row holds 64 MN elements (128 B),
// 8 K rows form a 1024-byte swizzle atom; "leading" byte offset = distance
// between 64-element MN blocks (one 64 x 64 box, 8 KB), "stride" byte offset
// = distance between 8-row K groups (1024 B).  One K = 16 step is 16 K rows,
// 2048 bytes further.
__device__ __forceinline__ uint64_t umma_desc_mn128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(kGemmBoxBytes >> 4) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

struct GemmArgs {
    int64_t M, N;             // output extent
    int nmb, nnb, nkb;        // blocks of 128 rows, 256 columns, 64 K
    int splits;               // K splits (>= 1)
    float* C;                 // [M, ldc] FP32 row-major; split s at C + s * split_stride
    int64_t ldc, split_stride;
    int accumulate;           // 1: C = C + A B (one rounding per element)
    int vec;                  // C rows 16-byte aligned (base and ldc)
};

struct GemmUnit {
    int s, mb, nb;
};

__device__ __forceinline__ GemmUnit gemm_unit(int64_t u, const GemmArgs& p) {
    const int64_t per = (int64_t)p.nmb * p.nnb;
    const int s = (int)(u / per);
    const int64_t t = u - (int64_t)s * per;
    return GemmUnit{s, (int)(t / p.nnb), (int)(t % p.nnb)};
}

// Loads of one K block of the A (or B) tile into `dst`: one K-major box of
// `rows` x 64, or rows/64 MN-major boxes of 64 x 64 placed 8 KB apart.
template <bool kMN, int kRows>
__device__ __forceinline__ void gemm_load(uint32_t dst, const CUtensorMap* map, int mn0, int k0, uint32_t bar) {
    if constexpr (kMN) {
#pragma unroll
        for (int j = 0; j < kRows / 64; ++j) tma_load_2d(dst + j * kGemmBoxBytes, map, mn0 + 64 * j, k0, bar);
    } else {
        tma_load_2d(dst, map, k0, mn0, bar);
    }
}

template <bool kMN>
__device__ __forceinline__ uint64_t gemm_desc(uint32_t addr) {
    if constexpr (kMN) return umma_desc_mn128(addr);
    else return umma_desc_swz(addr);
}

// K step of 16 inside a 64-wide K block, in 16-byte units of the address field.
template <bool kMN>
__host__ __device__ constexpr uint64_t gemm_kstep() {
    return kMN ? (2048 >> 4) : (32 >> 4);
}

template <bool kAmn, bool kBmn>
__global__ void __launch_bounds__(kGemmThreads, 1)
k_gemm_bf16(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, GemmArgs p) {
    extern __shared__ __align__(1024) unsigned char gemm_smem_raw[];
    const uint32_t raw = smem_u32(gemm_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t bars = base + kGemmStages * kGemmStageBytes;
    const uint32_t full0 = bars, empty0 = bars + 8 * kGemmStages;
    const uint32_t tfull0 = bars + 16 * kGemmStages, tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    const uint32_t slot = drain + 8;
    unsigned char* slot_gen = gemm_smem_raw + (slot - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(slot_gen);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slot_gen + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nunits = (int64_t)p.nmb * p.nnb * p.splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
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
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_b);
    }
    if (warp == 1) {
        tmem_alloc(slot, 2 * kGemmBN);
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
            for (int64_t u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
                const GemmUnit w = gemm_unit(u, p);
                const int kb0 = (int)((int64_t)w.s * p.nkb / p.splits);
                const int kb1 = (int)((int64_t)(w.s + 1) * p.nkb / p.splits);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!lin_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_dst = base + stage * kGemmStageBytes;
                    const uint32_t bar = full0 + 8 * stage;
                    mbar_arrive_expect_tx(bar, kGemmStageBytes);
                    gemm_load<kAmn, kGemmBM>(a_dst, &tm_a, w.mb * kGemmBM, kb * kGemmBK, bar);
                    gemm_load<kBmn, kGemmBN>(a_dst + kGemmABytes, &tm_b, w.nb * kGemmBN, kb * kGemmBK, bar);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == kGemmStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < kGemmStages; ++s)
                    if (issued & (1u << s)) mbar_wait(full0 + 8 * s, (last_par >> s) & 1u, kWaitLimitCycles);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = gemm_idesc<kAmn, kBmn>();
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
                const GemmUnit w = gemm_unit(u, p);
                const int kb0 = (int)((int64_t)w.s * p.nkb / p.splits);
                const int kb1 = (int)((int64_t)(w.s + 1) * p.nkb / p.splits);
                if (!lin_wait(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * kGemmBN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!lin_wait(full0 + 8 * stage, phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = base + stage * kGemmStageBytes;
                    const uint64_t a_desc = gemm_desc<kAmn>(a_addr);
                    const uint64_t b_desc = gemm_desc<kBmn>(a_addr + kGemmABytes);
#pragma unroll
                    for (int k = 0; k < kGemmBK / 16; ++k)
                        umma_bf16(d_tmem, a_desc + gemm_kstep<kAmn>() * k, b_desc + gemm_kstep<kBmn>() * k, idesc,
                                  (kb != kb0 || k != 0) ? 1u : 0u);
                    umma_commit(empty0 + 8 * stage);
                    if (++stage == kGemmStages) {
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
            umma_commit(drain);
            mbar_wait(drain, 0, kWaitLimitCycles);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: one output row per thread
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
            const GemmUnit w = gemm_unit(u, p);
            if (!lin_wait(tfull0 + 8 * acc, acc_phase, abort_flag)) break;
            tc_fence_after();
            const int64_t m = (int64_t)w.mb * kGemmBM + row;
            const int64_t n0 = (int64_t)w.nb * kGemmBN;
            float* crow = p.C + (int64_t)w.s * p.split_stride + m * p.ldc;
#pragma unroll 1
            for (int c = 0; c < kGemmBN / 32; ++c) {
                const int64_t c0 = n0 + c * 32;
                if (c0 >= p.N) break;   // uniform over the CTA
                __syncwarp();
                uint32_t r[32];
                tmem_ld32(lane_addr + (uint32_t)(acc * kGemmBN + c * 32), r);
                if (m < p.M) {
                    if (p.vec && c0 + 32 <= p.N) {
                        float4* dst = reinterpret_cast<float4*>(crow + c0);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float4 v = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                   __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                            if (p.accumulate) {
                                const float4 o = dst[j];
                                v.x = __fadd_rn(o.x, v.x);
                                v.y = __fadd_rn(o.y, v.y);
                                v.z = __fadd_rn(o.z, v.z);
                                v.w = __fadd_rn(o.w, v.w);
                            }
                            dst[j] = v;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (c0 + j < p.N) {
                                const float v = __uint_as_float(r[j]);
                                crow[c0 + j] = p.accumulate ? __fadd_rn(crow[c0 + j], v) : v;
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * kGemmBN);
    }
}

// Fixed-order sum of the K splits: out[r, c] = (((p_0 + p_1) + p_2) + ...)
// (+ out[r, c] first when accumulating) for rows [0, rows), columns [0, cols);
// the splits are [rows_total, cols] FP32 blocks split_stride apart.
__global__ void __launch_bounds__(256)
k_gemm_split_sum(const float* __restrict__ parts, int splits, int64_t split_stride, int64_t ldp, int64_t rows,
                 int64_t cols, float* __restrict__ out, int64_t ldo, int accumulate) {
    const int64_t total = rows * cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        const float* pp = parts + r * ldp + c;
        float s = accumulate ? out[r * ldo + c] : 0.f;
        float acc = __ldg(pp);
        for (int k = 1; k < splits; ++k) acc = __fadd_rn(acc, __ldg(pp + (int64_t)k * split_stride));
        out[r * ldo + c] = accumulate ? __fadd_rn(s, acc) : acc;
    }
}

}  // namespace flp
