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
    int64_t c_split_rows;     // tensor-map output: rows between consecutive splits
    int group;                // pair kernel: 0 = N blocks fastest; g > 0 = groups of g 256-row blocks, row block fastest
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

// ---------------------------------------------------------------- CTA pairs

// The same contraction on CTA pairs (a cluster of 2) with tcgen05.mma
// cta_group::2: a pair computes a 256 x 256 tile, each CTA holding 128 rows of
// A and 128 columns of B per K block (32 KB per stage instead of 48 KB, for
// the same FLOPs per SM), in a 6-stage ring.  Each CTA's producer copies its
// own halves of a stage into its own shared memory, completing on the even
// CTA's (rank 0) stage barrier, which expects both CTAs' bytes; the even CTA's
// MMA lane issues M = 256 MMAs that read both CTAs' halves, the accumulator
// rows split between the CTAs' TMEM, and each CTA's four epilogue warps read
// their 128 rows.  The MMA lane commits each released stage and each ready
// accumulator to the barriers of both CTAs (one commit per CTA); both CTAs'
// epilogue warps release an accumulator on the even CTA's barrier.  Every
// cross-CTA access is a barrier signal inside the pair.  (Forwarding the
// even CTA's signals to the peer through a waiting thread instead measured
// 2.4 times slower: the hand-off latency exceeds what 6 stages cover.)
constexpr int kPairStages = 6;
constexpr uint32_t kPairABytes = 128 * kGemmBK * 2;          // 16 KB: this CTA's A rows
constexpr uint32_t kPairBBytes = 128 * kGemmBK * 2;          // 16 KB: this CTA's B columns
constexpr uint32_t kPairStageBytes = kPairABytes + kPairBBytes;
// epilogue staging: per epilogue warp two 32 x 32 FP32 boxes (128-byte swizzle)
constexpr uint32_t kPairStageOutBytes = 32 * 32 * 4;
constexpr size_t kPairSmemBytes =
    1024 + (size_t)kPairStages * kPairStageBytes + 1024 + 4 * 2 * (size_t)kPairStageOutBytes;
static_assert(kPairSmemBytes <= 232448, "shared memory per CTA");

template <bool kAmn, bool kBmn>
__host__ __device__ constexpr uint32_t pair_idesc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((kAmn ? 1u : 0u) << 15) | ((kBmn ? 1u : 0u) << 16) |
           ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// The shared::cluster address of `addr` (a shared::cta address of this CTA)
// in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Bounded wait (cluster-scope acquire) that also gives up on the abort flag.
__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_cluster(bar, parity)) return true;
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
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Tensor-map store of a shared-memory box to global memory, or its addition
// to what global memory holds (the add is done where the data lives, one
// rounding per element); completion is tracked as a bulk group of this thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t x, int32_t y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, int32_t x, int32_t y, uint32_t src) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// At most N of this thread's bulk groups still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Loads of one K block of this pair's A (or B) half for CTA `rank` into its
// stage at `dst` (a shared::cluster address): 128 rows (K-major box) or two
// MN-major 64 x 64 boxes.
template <bool kMN>
__device__ __forceinline__ void pair_load(uint32_t dst, const CUtensorMap* map, int mn0, int k0, uint32_t bar) {
    if constexpr (kMN) {
        tma_load_2d_pair(dst, map, mn0, k0, bar);
        tma_load_2d_pair(dst + kGemmBoxBytes, map, mn0 + 64, k0, bar);
    } else {
        tma_load_2d_pair(dst, map, k0, mn0, bar);
    }
}

// kTmaC: the output goes out through tm_c (FP32 [rows, N], boxes of 32 x 32,
// 128-byte swizzle; split s at rows s * c_split_rows + m): each epilogue warp
// stages a 32 x 32 box in shared memory and one lane stores it, or adds it in
// place when accumulating, as whole lines.  Otherwise each thread writes its
// row's values itself.
template <bool kAmn, bool kBmn, bool kTmaC>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
k_gemm_bf16_pair(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_c, GemmArgs p) {
    extern __shared__ __align__(1024) unsigned char pair_smem_raw[];
    const uint32_t raw = smem_u32(pair_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // the same offset in both CTAs
    const uint32_t bars = base + kPairStages * kPairStageBytes;
    const uint32_t full0 = bars, empty0 = bars + 8 * kPairStages;
    const uint32_t tfull0 = bars + 16 * kPairStages, tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    const uint32_t slot = drain + 8;
    unsigned char* slot_gen = pair_smem_raw + (slot - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(slot_gen);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slot_gen + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    // this pair's units: (split, 256-row block, 256-column block), N fastest
    const int64_t nmb2 = (p.M + 255) / 256, nnb = p.nnb;
    const int64_t nunits = nmb2 * nnb * p.splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 8);     // 4 epilogue warps per CTA, both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_b);
        if (kTmaC) prefetch_tmap(&tm_c);
    }
    if (warp == 1) {
        tmem_alloc_pair(slot, 2 * kGemmBN);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto unit_of = [&](int64_t u, int& s, int64_t& mb, int64_t& nb) {
        const int64_t per = nmb2 * nnb;
        s = (int)(u / per);
        const int64_t t = u - (int64_t)s * per;
        if (p.group > 0) {   // groups of `group` row blocks: inside a group the row block is the fast index
            const int64_t gsz = (int64_t)p.group * nnb;
            const int64_t g = t / gsz, r = t - g * gsz;
            const int64_t rows = (g + 1) * p.group <= nmb2 ? p.group : nmb2 - g * p.group;
            mb = g * p.group + r % rows;
            nb = r / rows;
        } else {
            mb = t / nnb;
            nb = t - mb * nnb;
        }
    };

    if (warp == 0) {
        // ---------------- producers: each CTA copies its own halves of a stage;
        // every copy completes on the even CTA's stage barrier, which expects
        // both CTAs' bytes.  Each CTA's stage is released to its producer by
        // an MMA commit on its own barrier.
        if (lane == 0) {
            const uint32_t full_leader = map_to_rank(full0, 0);
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            bool ok = true;
            for (int64_t u = cid; ok && u < nunits; u += ncl) {
                int s;
                int64_t mb, nb;
                unit_of(u, s, mb, nb);
                const int kb0 = (int)((int64_t)s * p.nkb / p.splits);
                const int kb1 = (int)((int64_t)(s + 1) * p.nkb / p.splits);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!lin_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t off = stage * kPairStageBytes;
                    const uint32_t bar = full_leader + 8 * stage;
                    if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * kPairStageBytes);
                    const int k0 = kb * kGemmBK;
                    const int m0 = (int)(mb * 256) + (int)rank * 128, n0 = (int)(nb * 256) + (int)rank * 128;
                    pair_load<kAmn>(base + off, &tm_a, m0, k0, bar);
                    pair_load<kBmn>(base + off + kPairABytes, &tm_b, n0, k0, bar);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && leader) {
                for (int s = 0; s < kPairStages; ++s)
                    if (issued & (1u << s)) mbar_wait(full0 + 8 * s, (last_par >> s) & 1u, kWaitLimitCycles);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (even CTA): each commit is issued once
        // for this CTA's barrier and once for the peer's
        if (leader && lane == 0) {
            constexpr uint32_t idesc = pair_idesc<kAmn, kBmn>();
            const uint32_t empty_peer = map_to_rank(empty0, 1), tfull_peer = map_to_rank(tfull0, 1);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int64_t u = cid; ok && u < nunits; u += ncl) {
                int s;
                int64_t mb, nb;
                unit_of(u, s, mb, nb);
                const int kb0 = (int)((int64_t)s * p.nkb / p.splits);
                const int kb1 = (int)((int64_t)(s + 1) * p.nkb / p.splits);
                // both CTAs' epilogues have released this accumulator
                if (!pair_wait(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag)) {
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
                    const uint32_t a_addr = base + stage * kPairStageBytes;
                    const uint64_t a_desc = gemm_desc<kAmn>(a_addr);
                    const uint64_t b_desc = gemm_desc<kBmn>(a_addr + kPairABytes);
#pragma unroll
                    for (int k = 0; k < kGemmBK / 16; ++k)
                        umma_bf16_pair(d_tmem, a_desc + gemm_kstep<kAmn>() * k, b_desc + gemm_kstep<kBmn>() * k,
                                       idesc, (kb != kb0 || k != 0) ? 1u : 0u);
                    umma_commit_pair(empty0 + 8 * stage);
                    umma_commit_pair(empty_peer + 8 * stage);
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(tfull0 + 8 * acc);
                umma_commit_pair(tfull_peer + 8 * acc);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            umma_commit_pair(drain);
            mbar_wait(drain, 0, kWaitLimitCycles);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: this CTA's 128 rows of the pair's tile
        const int q = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
        const uint32_t tempty_leader = map_to_rank(tempty0, 0);
        const uint32_t stg = bars + 1024 + (uint32_t)q * 2 * kPairStageOutBytes;   // this warp's two boxes
        int acc = 0, nbuf = 0;
        uint32_t acc_phase = 0;
        for (int64_t u = cid; u < nunits; u += ncl) {
            int s;
            int64_t mb, nb;
            unit_of(u, s, mb, nb);
            if (!lin_wait(tfull0 + 8 * acc, acc_phase, abort_flag)) break;
            tc_fence_after();
            const int64_t m_warp = mb * 256 + (int64_t)rank * 128 + q * 32;   // first row of this warp
            const int64_t m = m_warp + lane;
            const int64_t n0 = nb * kGemmBN;
            float* crow = p.C + (int64_t)s * p.split_stride + m * p.ldc;
#pragma unroll 1
            for (int c = 0; c < kGemmBN / 32; ++c) {
                const int64_t c0 = n0 + c * 32;
                if (c0 >= p.N) break;   // uniform over the CTA
                __syncwarp();
                if constexpr (kTmaC) {
                    uint32_t r[32];
                    tmem_ld32(lane_addr + (uint32_t)(acc * kGemmBN + c * 32), r);
                    if (m_warp >= p.M) continue;   // the whole box lies past the last row
                    const uint32_t box = stg + (uint32_t)(nbuf & 1) * kPairStageOutBytes;
                    if (lane == 0) bulk_wait_read<1>();   // the store that last used this box has read it
                    __syncwarp();
                    // row `lane` of the box, 16-byte chunk j at position j ^ (lane mod 8)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        sts_v4(box + (uint32_t)lane * 128 + (uint32_t)((j ^ (lane & 7)) * 16), r[4 * j], r[4 * j + 1],
                               r[4 * j + 2], r[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int32_t y = (int32_t)((int64_t)s * p.c_split_rows + m_warp);
                        if (p.accumulate) tma_reduce_add_2d(&tm_c, (int32_t)c0, y, box);
                        else tma_store_2d(&tm_c, (int32_t)c0, y, box);
                        bulk_commit_group();
                    }
                    ++nbuf;
                } else {
                    const bool vec = p.vec && c0 + 32 <= p.N && m < p.M;
                    float4 old[8];
                    if (vec && p.accumulate) {
                        const float4* src = reinterpret_cast<const float4*>(crow + c0);
#pragma unroll
                        for (int j = 0; j < 8; ++j) old[j] = src[j];
                    }
                    uint32_t r[32];
                    tmem_ld32(lane_addr + (uint32_t)(acc * kGemmBN + c * 32), r);
                    if (vec) {
                        float4* dst = reinterpret_cast<float4*>(crow + c0);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float4 v = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                   __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                            if (p.accumulate) {
                                v.x = __fadd_rn(old[j].x, v.x);
                                v.y = __fadd_rn(old[j].y, v.y);
                                v.z = __fadd_rn(old[j].z, v.z);
                                v.w = __fadd_rn(old[j].w, v.w);
                            }
                            dst[j] = v;
                        }
                    } else if (m < p.M) {
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
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + 8 * acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (kTmaC && lane == 0) bulk_wait_read<0>();   // shared memory is read before the CTA exits
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // no copy, arrive or MMA of the pair still targets either CTA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 2 * kGemmBN);
    }
}

}  // namespace flp
