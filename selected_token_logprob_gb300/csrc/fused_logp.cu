// Host side of libfused_logp.so: argument checks, device guard, launch
// configuration and the extern "C" entry points declared in
// include/fused_logp.h.  All checks run on the host before any launch and
// report through the return code (no device-side traps).
#include <cuda_runtime.h>
#include <math.h>

#include <atomic>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "fused_logp.h"
#include "gemm_bf16.cuh"
#include "grpo_kernels.cuh"
#include "linear_logp.cuh"
#include "logp_kernels.cuh"

// Fixed device scratch of fused_linear_logp_forward_noalloc, for callers that
// cannot allocate device memory.  It lives in the module's static device
// memory: every GPU that loads this library holds these 16 MiB until the
// process exits.  Host code must not pass this name to a kernel (on the host
// it names a stand-in object, not device memory); it looks up the device
// address once per device with cudaGetSymbolAddress.
constexpr int64_t kNoAllocScratchBytes = (int64_t)16 << 20;
static __device__ __align__(256) float g_linear_noalloc_scratch[kNoAllocScratchBytes / 4];

namespace {

thread_local char g_msg[512] = "";

flp_status fail(flp_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

flp_status ok() {
    g_msg[0] = '\0';
    return FLP_OK;
}

int64_t tile_width(int64_t v) {
    if (v < 1) return 0;
    const int64_t per = flp::kTiles * 8;
    return 8 * ((v + per - 1) / per);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int elem_bytes(int dtype) { return dtype == FLP_DTYPE_F32 ? 4 : 2; }

// Bytes spanned by an [n, ld] matrix whose rows use the first `v` columns.
bool span_bytes(int64_t n, int64_t v, int64_t ld, int64_t elem, int64_t* out) {
    int64_t a, b;
    if (__builtin_mul_overflow(n - 1, ld, &a)) return false;
    if (__builtin_add_overflow(a, v, &b)) return false;
    if (__builtin_mul_overflow(b, elem, out)) return false;
    return true;
}

// Device that holds `p`; FLP_EINVAL if `p` is not device-accessible memory.
flp_status device_of(const void* p, const char* name, int* dev) {
    if (p == nullptr) return fail(FLP_EINVAL, "%s is a null pointer", name);
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail(FLP_EINVAL, "%s: cudaPointerGetAttributes failed (%s)", name, cudaGetErrorString(e));
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
        return fail(FLP_EINVAL, "%s must point to device memory", name);
    *dev = a.device;
    return FLP_OK;
}

// Every required pointer, and every optional one that is not null, must be
// device memory of one device; returns that device.
flp_status common_device(int count, const void* const* ptrs, const char* const* names,
                         const bool* optional, int* dev) {
    int d0 = -1;
    const char* first = nullptr;
    for (int i = 0; i < count; ++i) {
        if (optional && optional[i] && ptrs[i] == nullptr) continue;
        int d;
        const flp_status st = device_of(ptrs[i], names[i], &d);
        if (st != FLP_OK) return st;
        if (!first) {
            d0 = d;
            first = names[i];
        } else if (d != d0) {
            return fail(FLP_EINVAL, "%s is on device %d but %s is on device %d", names[i], d, first, d0);
        }
    }
    *dev = d0;
    return FLP_OK;
}

// Makes `dev` current for the call and restores the caller's device after.
struct DeviceGuard {
    int prev = -1;
    bool switched = false;
    flp_status enter(int dev) {
        cudaError_t e = cudaGetDevice(&prev);
        if (e != cudaSuccess) return fail(FLP_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
        if (prev != dev) {
            e = cudaSetDevice(dev);
            if (e != cudaSuccess) return fail(FLP_ECUDA, "cudaSetDevice: %s", cudaGetErrorString(e));
            switched = true;
        }
        return FLP_OK;
    }
    ~DeviceGuard() {
        if (switched) (void)cudaSetDevice(prev);
    }
};

flp_status check_launch(const char* what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FLP_ECUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
    return ok();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rows start on 16-byte boundaries: base aligned and the byte stride a
// multiple of 16.
bool rows_aligned16(const void* p, int64_t ld, int dtype) {
    return aligned16(p) && (ld * elem_bytes(dtype)) % 16 == 0;
}

constexpr int64_t kMaxGrid = 2147483647;
constexpr int kMaxDevices = 64;

int grid_for(int64_t items) { return (int)(items < kMaxGrid ? items : kMaxGrid); }

flp_status check_dtype(int dtype) {
    if (dtype != FLP_DTYPE_BF16 && dtype != FLP_DTYPE_F16 && dtype != FLP_DTYPE_F32)
        return fail(FLP_EINVAL, "dtype must be FLP_DTYPE_BF16, FLP_DTYPE_F16 or FLP_DTYPE_F32 (got %d)", dtype);
    return FLP_OK;
}

flp_status check_scale(float s) {
    if (!(s > 0.f) || !isfinite(s))
        return fail(FLP_EINVAL, "inv_temperature must be finite and > 0 (got %g)", (double)s);
    return FLP_OK;
}

// s and s log2(e) as a two-float hi + lo, from the double value of log2(e).
// hi is rounded down and lo kept strictly positive, so that t hi + t lo is
// -inf (never -inf + inf = NaN) for a -inf logit difference t.
flp::Scale make_scale(float s) {
    const double c = (double)s * 1.4426950408889634073599246810019;
    float hi = (float)c;
    if ((double)hi > c) hi = nextafterf(hi, 0.f);
    float lo = (float)(c - (double)hi);
    if (!(lo > 0.f)) lo = 1e-30f;
    return flp::Scale{s, hi, lo};
}

// Per-device caches below are atomics: host threads may call in
// concurrently; every writer stores the same value, so the first one wins.
int sm_count(int dev) {
    static std::atomic<int> count[kMaxDevices];
    int c = count[dev].load(std::memory_order_acquire);
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        count[dev].store(c, std::memory_order_release);
    }
    return c;
}

// Once per device and kernel: allow the bulk-copy forward its dynamic shared
// memory (idempotent, so two threads doing it at once is harmless).
template <flp::Dt D, bool kScaled>
flp_status bulk_setup(int dev) {
    static std::atomic<bool> ready[kMaxDevices];
    if (!ready[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(flp::k_logp_fwd_bulk<D, kScaled>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   flp::kFwdSmemBytes<D>);
        if (e != cudaSuccess) return fail(FLP_ECUDA, "forward setup: %s", cudaGetErrorString(e));
        ready[dev].store(true, std::memory_order_release);
    }
    return FLP_OK;
}

struct FwdArgs {
    const void* x;
    int64_t n, v, ld, W;
    const int64_t* y;
    int64_t ii;
    const uint8_t* mask;
    flp::Scale sc;
    float *logp, *lse, *lse_lo;
    cudaStream_t s;
    int dev;
    bool bulk;
};

template <flp::Dt D, bool kScaled>
flp_status launch_forward(const FwdArgs& a) {
    if (a.bulk) {
        flp_status st = bulk_setup<D, kScaled>(a.dev);
        if (st != FLP_OK) return st;
        const int sms = sm_count(a.dev);
        if (sms <= 0) return fail(FLP_ECUDA, "could not read the SM count of device %d", a.dev);
        const int64_t ctas = (int64_t)flp::kFwdMinBlocks<D> * sms;
        const int grid = grid_for(a.n < ctas ? a.n : ctas);
        flp::k_logp_fwd_bulk<D, kScaled><<<grid, flp::kFwdThreads, flp::kFwdSmemBytes<D>, a.s>>>(
            a.x, a.n, a.v, a.ld, a.W, a.y, a.ii, a.mask, a.sc, a.logp, a.lse, a.lse_lo);
    } else {
        flp::k_logp_fwd<D, kScaled><<<grid_for(a.n), flp::kFwdThreads, 0, a.s>>>(
            a.x, a.n, a.v, a.ld, a.W, a.y, a.ii, a.mask, a.sc, a.logp, a.lse, a.lse_lo);
    }
    return check_launch("forward");
}

// The exponent argument always uses the two-float s log2(e) (also at s = 1,
// where it removes the rounding of log2(e) to binary32 from every term).
template <flp::Dt D>
flp_status launch_forward_d(const FwdArgs& a) {
    return launch_forward<D, true>(a);
}

struct BwdArgs {
    const void* x;
    int64_t n, v, ld;
    const int64_t* y;
    int64_t ii;
    const uint8_t* mask;
    float s, inv_s;
    const float *lse, *lse_lo, *g;
    void* dx;
    int64_t ld_out;
    cudaStream_t st;
    bool vin, vout, in_place;
    int64_t y_off, v_total;   // the buffer's first global column; the whole vocabulary
};

template <flp::Dt D, bool VI, bool VO, bool IP>
void launch_bwd(const BwdArgs& a, dim3 grid) {
    flp::k_logp_bwd<D, VI, VO, IP><<<grid, flp::kBwdThreads, 0, a.st>>>(
        a.x, a.n, a.v, a.ld, a.y, a.ii, a.mask, a.s, a.inv_s, a.lse, a.lse_lo, a.g, a.dx, a.ld_out, a.y_off,
        a.v_total);
}

template <flp::Dt D>
void launch_backward_d(const BwdArgs& a, dim3 grid) {
    if (a.in_place) {
        if (a.vin) launch_bwd<D, true, true, true>(a, grid);
        else launch_bwd<D, false, false, true>(a, grid);
    } else if (a.vin && a.vout) launch_bwd<D, true, true, false>(a, grid);
    else if (a.vin) launch_bwd<D, true, false, false>(a, grid);
    else if (a.vout) launch_bwd<D, false, true, false>(a, grid);
    else launch_bwd<D, false, false, false>(a, grid);
}

struct PartArgs {
    const void* xs;
    int64_t n, ld, real_width, W;
    int tile0, ntile;
    int64_t vocab_start;
    const int64_t* y;
    flp::Scale sc;
    float *pm, *ps, *sel;
    cudaStream_t s;
    bool vec;
};

template <flp::Dt D, bool V, bool S>
void launch_part(const PartArgs& a) {
    flp::k_logp_partials<D, V, S><<<grid_for(a.n), a.ntile * flp::kWarp, 0, a.s>>>(
        a.xs, a.n, a.ld, a.real_width, a.W, a.tile0, a.vocab_start, a.y, a.sc, a.pm, a.ps, a.sel);
}

template <flp::Dt D>
void launch_partials_d(const PartArgs& a) {
    if (a.vec) launch_part<D, true, true>(a);
    else launch_part<D, false, true>(a);
}

// ---- fused LM head: tensor maps and launch setup

// cuTensorMapEncodeTiled from the driver, found once through the runtime (no
// link against the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            (void)cudaGetLastError();
            return (EncodeTiledFn) nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// Tensor map of a BF16 row-major [rows, ld] matrix whose first `cols` columns
// are used: boxes of kLinBK columns (one swizzle span) x box_rows rows, the
// swizzle the contraction kernel's descriptors expect, zero fill outside the
// matrix.
flp_status make_tmap_bf16(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                          uint32_t box_rows, const char* name) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return fail(FLP_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {(cuuint32_t)flp::kLinBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          flp::kLinRowBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FLP_EINVAL, "tensor map of %s rejected by the driver (error %d)", name, (int)r);
    return FLP_OK;
}

// Tensor map of an FP32 row-major [rows, ld] output matrix whose first `cols`
// columns are written: boxes of 32 x 32 with 128-byte swizzle (the layout the
// contraction's epilogue stages).  False when the layout does not allow one
// (base not 16-byte aligned, row stride not a multiple of 16 bytes).
bool make_tmap_f32_out(CUtensorMap* m, void* ptr, int64_t rows, int64_t cols, int64_t ld) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn || !aligned16(ptr) || (ld * 4) % 16 != 0 || rows < 1 || cols < 1) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

flp_status linear_setup(int dev) {
    static std::atomic<bool> ready[kMaxDevices];
    if (!ready[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(flp::k_linear_logp_tiles<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)flp::kLinSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(flp::k_linear_logp_tiles<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)flp::kLinSmemBytes);
        if (e != cudaSuccess) return fail(FLP_ECUDA, "linear logp setup: %s", cudaGetErrorString(e));
        ready[dev].store(true, std::memory_order_release);
    }
    return FLP_OK;
}

// ---- fused LM head backward: row chunks and the two tensor-core products

// Rows per chunk of the backward: dZ is materialised for one chunk at a time.
// Every row's dZ and dH are computed the same way whatever the chunk holds.
constexpr int64_t kLinGradChunk = 4096;
// K blocks of 64 per split of the dH product (K = the vocabulary): enough
// splits that the (split, tile) units fill the SMs in near-whole waves.
constexpr int64_t kGemmSplitKBlocks = 512;

int64_t align256(int64_t b) { return ceil_div(b, 256) * 256; }

// K splits of dH = dZ W for a v-column vocabulary: a function of v only.
int dh_splits(int64_t v) {
    const int64_t s = ceil_div(ceil_div(v, flp::kGemmBK), kGemmSplitKBlocks);
    return (int)(s < 1 ? 1 : s);
}

// Backward workspace: dZ [chunk, ld_dz] BF16, then (with more than one K
// split) the splits' partial dH [splits, chunk, d] FP32.
bool linear_grad_workspace(int64_t d, int64_t v, int64_t* ld_dz, int64_t* off_dh, int64_t* total) {
    const int64_t ld = ceil_div(v, 8) * 8;
    const int64_t splits = dh_splits(v);
    int64_t a, b = 0;
    if (__builtin_mul_overflow(kLinGradChunk, ld, &a) || __builtin_mul_overflow(a, (int64_t)2, &a)) return false;
    if (splits > 1 && (__builtin_mul_overflow(kLinGradChunk, d, &b) || __builtin_mul_overflow(b, splits * 4, &b)))
        return false;
    *ld_dz = ld;
    *off_dh = align256(a);
    *total = *off_dh + align256(b);
    return true;
}

flp_status gemm_setup(int dev) {
    static std::atomic<bool> ready[kMaxDevices];
    if (!ready[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(flp::k_gemm_bf16<false, true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)flp::kGemmSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(flp::k_gemm_bf16<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)flp::kGemmSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(flp::k_gemm_bf16_pair<false, true, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)flp::kPairSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(flp::k_gemm_bf16_pair<true, true, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)flp::kPairSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(flp::k_gemm_bf16_pair<false, true, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)flp::kPairSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(flp::k_gemm_bf16_pair<true, true, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)flp::kPairSmemBytes);
        if (e != cudaSuccess) return fail(FLP_ECUDA, "contraction setup: %s", cudaGetErrorString(e));
        ready[dev].store(true, std::memory_order_release);
    }
    return FLP_OK;
}

// C (+)= A B on the tensor cores: M x N output, K-extent k, `splits` K splits
// written split_stride floats apart.  CTA pairs (tcgen05 cta_group::2) when a
// pair fits on the device, else one CTA per 128 x 256 tile (same bits).  A is K-major (kAmn = false) or MN-major,
// B is MN-major; the tensor maps carry the operands' layouts.
// Clusters of the pair kernel that can be resident at once on `dev` (cached).
template <bool kAmn>
int pair_clusters(int dev) {
    static std::atomic<int> count[kMaxDevices];
    int c = count[dev].load(std::memory_order_acquire);
    if (c == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(flp::kGemmThreads);
        cfg.dynamicSmemBytes = flp::kPairSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&c, (void*)flp::k_gemm_bf16_pair<kAmn, true, true>, &cfg) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        count[dev].store(c, std::memory_order_release);
    }
    return c;
}

template <bool kAmn>
flp_status gemm_launch(int dev, int sms, const CUtensorMap& tm_a, const CUtensorMap& tm_b, int64_t m, int64_t n,
                       int64_t k, int splits, float* c, int64_t ldc, int64_t split_stride, int64_t c_rows,
                       bool accumulate, cudaStream_t s, const char* what) {
    flp::GemmArgs g;
    g.M = m;
    g.N = n;
    g.nmb = (int)ceil_div(m, flp::kGemmBM);
    g.nnb = (int)ceil_div(n, flp::kGemmBN);
    g.nkb = (int)ceil_div(k, flp::kGemmBK);
    g.splits = splits;
    g.C = c;
    g.ldc = ldc;
    g.split_stride = split_stride;
    g.accumulate = accumulate ? 1 : 0;
    g.vec = (aligned16(c) && ldc % 4 == 0 && split_stride % 4 == 0) ? 1 : 0;
    g.c_split_rows = (splits > 1 && ldc > 0) ? split_stride / ldc : 0;
    g.group = 0;
    const int fit = pair_clusters<kAmn>(dev);
    if (fit > 0) {
        // CTA pairs: a 256 x 256 tile per pair, as many pairs as fit at once; the
        // output leaves through a tensor map of C (all splits' rows) when C allows one
        const int64_t units = ceil_div(m, 256) * g.nnb * splits;
        const int64_t pairs = units < fit ? units : fit;
        CUtensorMap tm_c;
        const bool tma_c = (splits == 1 || split_stride % ldc == 0) &&
                           make_tmap_f32_out(&tm_c, c, splits > 1 ? g.c_split_rows * splits : c_rows, n, ldc);
        if (tma_c)
            flp::k_gemm_bf16_pair<kAmn, true, true><<<(int)(2 * pairs), flp::kGemmThreads, flp::kPairSmemBytes, s>>>(
                tm_a, tm_b, tm_c, g);
        else
            flp::k_gemm_bf16_pair<kAmn, true, false><<<(int)(2 * pairs), flp::kGemmThreads, flp::kPairSmemBytes, s>>>(
                tm_a, tm_b, tm_a, g);
        return check_launch(what);
    }
    const int64_t units = (int64_t)g.nmb * g.nnb * splits;
    const int grid = (int)(units < sms ? units : sms);
    flp::k_gemm_bf16<kAmn, true><<<grid, flp::kGemmThreads, flp::kGemmSmemBytes, s>>>(tm_a, tm_b, g);
    return check_launch(what);
}

int64_t linear_vocab_tiles(int64_t v) { return ceil_div(v, flp::kLinBN); }

// Workspace: tile maxima [n, nvt], tile sums [n, nvt], selected logits [n]
// (binary32), rounded up to 256 bytes; false on overflow.
bool linear_workspace_bytes(int64_t n, int64_t v, int64_t* out) {
    int64_t a, b;
    if (__builtin_mul_overflow(linear_vocab_tiles(v), n, &a)) return false;
    if (__builtin_mul_overflow(a, (int64_t)2, &a)) return false;
    if (__builtin_add_overflow(a, n, &b)) return false;
    if (__builtin_mul_overflow(b, (int64_t)4, &b)) return false;
    *out = ceil_div(b, 256) * 256;
    return true;
}

// Device address of g_linear_noalloc_scratch on `dev` (which must be
// current), looked up on the first call for that device and cached (an
// atomic per device: concurrent first calls each look it up and store the
// same address).  The cached address belongs to the device's current
// context; after cudaDeviceReset it is stale.
flp_status noalloc_scratch_address(int dev, void** out) {
    static std::atomic<void*> addr[kMaxDevices];
    void* p = addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        const cudaError_t e = cudaGetSymbolAddress(&p, g_linear_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return fail(FLP_ECUDA, "address of the static scratch on device %d: %s", dev, cudaGetErrorString(e));
        }
        addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return FLP_OK;
}

// Tile partials of rows [0, n) against `weight` (w rows: global vocabulary
// columns [vocab_start, vocab_start + w), vocab_start on the 256-column tile
// grid) into the [n, ceil(v_total / 256)] partial buffers of `ws`, and the
// selected logit of every row whose target falls in those columns.
flp_status linear_partials_launch(int dev, const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                  const void* weight, int64_t w, int64_t ld_w, int64_t vocab_start, int64_t v_total,
                                  const int64_t* targets, int64_t ignore_index, const uint8_t* mask, float inv_s,
                                  float* ws, cudaStream_t stream) {
    flp_status st;
    if ((st = linear_setup(dev)) != FLP_OK) return st;
    CUtensorMap tm_h, tm_w;
    if ((st = make_tmap_bf16(&tm_h, hidden, n, d, ld_h, flp::kLinBM, "hidden")) != FLP_OK) return st;
    if ((st = make_tmap_bf16(&tm_w, weight, w, d, ld_w, flp::kLinBN, "weight")) != FLP_OK) return st;
    const int64_t nvt = linear_vocab_tiles(w);
    const int64_t nvt_total = linear_vocab_tiles(v_total);
    const int64_t nrb = ceil_div(n, flp::kLinBM);
    flp::LinArgs a;
    a.n = n;
    a.v = w;
    a.nrb = (int)nrb;
    a.nvt = (int)nvt;
    a.nkb = (int)ceil_div(d, flp::kLinBK);
    a.vocab_start = vocab_start;
    a.v_total = v_total;
    a.vt0 = (int)(vocab_start / flp::kLinBN);
    a.nvt_total = (int)nvt_total;
    a.y = targets;
    a.ignore_index = ignore_index;
    a.mask = mask;
    a.sc = make_scale(inv_s);
    a.pm = ws;
    a.ps = ws + nvt_total * n;
    a.xsel = ws + 2 * nvt_total * n;
    a.n_valid = n;
    a.lse = nullptr;
    a.lse_lo = nullptr;
    a.g = nullptr;
    a.inv_s = 0.f;
    a.dz = nullptr;
    a.ld_dz = 0;
    const int sms = sm_count(dev);
    if (sms <= 0) return fail(FLP_ECUDA, "cannot read the SM count of device %d", dev);
    const int64_t ntiles = nrb * nvt;
    const int grid = (int)(ntiles < sms ? ntiles : sms);
    flp::k_linear_logp_tiles<false><<<grid, flp::kLinThreads, flp::kLinSmemBytes, stream>>>(tm_h, tm_w, a);
    return check_launch("linear logp tiles");
}

// The fixed-order merge of the [n, ceil(v_total / 256)] partials in `ws`.
flp_status linear_merge_launch(int dev, const float* ws, int64_t n, int64_t v_total, const int64_t* targets,
                               int64_t ignore_index, const uint8_t* mask, float inv_s, float* logp, float* lse,
                               float* lse_lo, cudaStream_t stream) {
    const int64_t nvt_total = linear_vocab_tiles(v_total);
    const int sms = sm_count(dev);
    if (sms <= 0) return fail(FLP_ECUDA, "cannot read the SM count of device %d", dev);
    // one warp per row, at most 16 resident CTAs of 256 threads per SM
    const int64_t ctas = ceil_div(n * 32, flp::kLinMergeThreads);
    flp::k_linear_logp_merge<<<(int)(ctas < (int64_t)sms * 16 ? ctas : (int64_t)sms * 16), flp::kLinMergeThreads,
                               0, stream>>>(ws, ws + nvt_total * n, ws + 2 * nvt_total * n, n, (int)nvt_total,
                                            v_total, targets, ignore_index, mask, inv_s, logp, lse, lse_lo);
    return check_launch("linear logp merge");
}

// Launches kern<<<grid, block, 0, s>>>(args...) with programmatic stream
// serialization: the kernel may start while the previous work on s runs and
// waits for it with griddepcontrol.wait.
template <class... Args>
flp_status launch_dependent(const char* what, void (*kern)(Args...), int grid, int block, cudaStream_t s,
                            Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) return fail(FLP_ECUDA, "%s launch: %s", what, cudaGetErrorString(e));
    return ok();
}

// GRPO workspace: 32 bytes for the active-token count and the fold's
// ticket, two two-float sums per CTA of the token pass (608 CTAs), a count
// per CTA of the sequences' counts (1024) and per count range (1024), and
// with sequences two floats per sequence and a 32-bit word prefix per 16
// tokens; rounded up to 256 bytes.
int64_t grpo_workspace_bytes(int64_t n, int64_t nseq) {
    const int64_t seq_part = nseq > 0 ? 8 * nseq + 4 * ceil_div(n, 16) : 0;
    return ceil_div(32 + 16 * flp::kGrpoPassCtas + 8 * flp::kGrpoFixMaxCtas + 8 * flp::kGrpoCountMaxCtas + seq_part,
                    256) * 256;
}

}  // namespace

extern "C" {

const char* flp_last_error(void) { return g_msg; }

const char* flp_version(void) { return "fused_logp 0.2 (sm_103a)"; }

int64_t flp_tile_width(int64_t v) { return tile_width(v); }

flp_status fused_logp_forward_ex(const void* logits, int dtype, int64_t n, int64_t v, int64_t ld,
                                 const int64_t* targets, int64_t ignore_index,
                                 const uint8_t* active_mask, float inv_temperature, float* logp,
                                 float* lse, float* lse_lo, flp_stream_t stream) {
    flp_status st;
    if ((st = check_dtype(dtype)) != FLP_OK) return st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v < 1) return fail(FLP_EINVAL, "v must be >= 1 (got %lld)", (long long)v);
    if (ld < v) return fail(FLP_EINVAL, "ld (%lld) must be >= v (%lld)", (long long)ld, (long long)v);
    if (n == 0) return ok();
    int64_t bytes;
    if (!span_bytes(n, v, ld, elem_bytes(dtype), &bytes))
        return fail(FLP_EINVAL, "logits extent overflows int64");
    const void* ptrs[] = {logits, targets, logp, lse, lse_lo, active_mask};
    const char* names[] = {"logits", "targets", "logp", "lse", "lse_lo", "active_mask"};
    const bool optional[] = {false, false, false, false, true, true};
    int dev;
    if ((st = common_device(6, ptrs, names, optional, &dev)) != FLP_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;

    const FwdArgs a{logits, n, v, ld, tile_width(v), targets, ignore_index, active_mask,
                    make_scale(inv_temperature), logp, lse, lse_lo,
                    reinterpret_cast<cudaStream_t>(stream), dev,
                    rows_aligned16(logits, ld, dtype) && v < ((int64_t)1 << 31)};
    if (dtype == FLP_DTYPE_BF16) return launch_forward_d<flp::Dt::BF16>(a);
    if (dtype == FLP_DTYPE_F16) return launch_forward_d<flp::Dt::F16>(a);
    return launch_forward_d<flp::Dt::F32>(a);
}

flp_status fused_logp_forward(const void* logits, int64_t n, int64_t v, int64_t ld,
                              const int64_t* targets, int64_t ignore_index, float* logp,
                              float* lse, float* lse_lo, flp_stream_t stream) {
    return fused_logp_forward_ex(logits, FLP_DTYPE_BF16, n, v, ld, targets, ignore_index, nullptr,
                                 1.f, logp, lse, lse_lo, stream);
}

}  // extern "C"

namespace {

// The backward over a buffer of columns [y_off, y_off + v) of a
// v_total-column vocabulary (unsharded: 0 and v).
flp_status backward_impl(const void* logits, int dtype, int64_t n, int64_t v, int64_t ld, int64_t y_off,
                         int64_t v_total, const int64_t* targets, int64_t ignore_index,
                         const uint8_t* active_mask, float inv_temperature, const float* lse,
                         const float* lse_lo, const float* grad, void* dlogits, int64_t ld_out,
                         flp_stream_t stream) {
    flp_status st;
    if ((st = check_dtype(dtype)) != FLP_OK) return st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v < 1) return fail(FLP_EINVAL, "v must be >= 1 (got %lld)", (long long)v);
    if (y_off < 0 || y_off > v_total - v)
        return fail(FLP_EINVAL, "the columns [%lld, %lld) must lie inside the vocabulary [0, %lld)",
                    (long long)y_off, (long long)(y_off + v), (long long)v_total);
    if (ld < v) return fail(FLP_EINVAL, "ld (%lld) must be >= v (%lld)", (long long)ld, (long long)v);
    if (ld_out < v)
        return fail(FLP_EINVAL, "ld_out (%lld) must be >= v (%lld)", (long long)ld_out, (long long)v);
    if (n == 0) return ok();
    const int eb = elem_bytes(dtype);
    int64_t in_bytes, out_bytes;
    if (!span_bytes(n, v, ld, eb, &in_bytes) || !span_bytes(n, v, ld_out, eb, &out_bytes))
        return fail(FLP_EINVAL, "logits/dlogits extent overflows int64");
    const void* ptrs[] = {logits, targets, lse, grad, dlogits, lse_lo, active_mask};
    const char* names[] = {"logits", "targets", "lse", "grad", "dlogits", "lse_lo", "active_mask"};
    const bool optional[] = {false, false, false, false, false, true, true};
    int dev;
    if ((st = common_device(7, ptrs, names, optional, &dev)) != FLP_OK) return st;

    const uintptr_t xb = reinterpret_cast<uintptr_t>(logits);
    const uintptr_t db = reinterpret_cast<uintptr_t>(dlogits);
    const bool in_place = (xb == db) && (ld == ld_out);
    if (!in_place && xb < db + (uintptr_t)out_bytes && db < xb + (uintptr_t)in_bytes)
        return fail(FLP_EINVAL, "dlogits overlaps logits without being exactly in place");

    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;

    const int64_t segs = ceil_div(v, flp::kBwdSegCols);
    if (segs > kMaxGrid) return fail(FLP_EINVAL, "v too large for the backward grid");
    const BwdArgs a{logits, n, v, ld, targets, ignore_index, active_mask, inv_temperature,
                    1.f / inv_temperature, lse, lse_lo, grad, dlogits, ld_out,
                    reinterpret_cast<cudaStream_t>(stream), rows_aligned16(logits, ld, dtype),
                    rows_aligned16(dlogits, ld_out, dtype), in_place, y_off, v_total};
    const dim3 grid((unsigned)segs, (unsigned)(n < 65535 ? n : 65535));
    if (dtype == FLP_DTYPE_BF16) launch_backward_d<flp::Dt::BF16>(a, grid);
    else if (dtype == FLP_DTYPE_F16) launch_backward_d<flp::Dt::F16>(a, grid);
    else launch_backward_d<flp::Dt::F32>(a, grid);
    return check_launch("backward");
}

// Tile -> rank table of a vocabulary-parallel group: 4 bits per tile.  Every
// rank's shard must lie on the tile grid, and together they must cover each
// of the ceil(v_total / W) tiles exactly once.
flp_status tile_rank_table(int64_t world, const int64_t* starts, const int64_t* widths, int64_t v_total,
                           uint64_t* table) {
    if (world < 1 || world > flp::kTiles)
        return fail(FLP_EINVAL, "world must be in [1, %d] (got %lld)", flp::kTiles, (long long)world);
    if (starts == nullptr || widths == nullptr) return fail(FLP_EINVAL, "vocab_starts and real_widths are null");
    const int64_t W = tile_width(v_total);
    const int64_t n_tiles = ceil_div(v_total, W);
    int owner[flp::kTiles];
    for (int k = 0; k < flp::kTiles; ++k) owner[k] = -1;
    for (int64_t r = 0; r < world; ++r) {
        const int64_t a = starts[r], w = widths[r];
        if (w < 1 || a < 0 || a > v_total - w)
            return fail(FLP_EINVAL, "rank %lld: shard [%lld, %lld) is not inside [0, %lld)", (long long)r,
                        (long long)a, (long long)(a + w), (long long)v_total);
        if (a % W != 0 || (a + w != v_total && w % W != 0))
            return fail(FLP_EUNSUPPORTED, "rank %lld: shard [%lld, %lld) is off the %lld-column tile grid",
                        (long long)r, (long long)a, (long long)(a + w), (long long)W);
        for (int64_t k = a / W; k < ceil_div(a + w, W); ++k) {
            if (owner[k] >= 0)
                return fail(FLP_EINVAL, "tile %lld is held by rank %d and rank %lld", (long long)k, owner[k],
                            (long long)r);
            owner[k] = (int)r;
        }
    }
    uint64_t t = 0;
    for (int64_t k = 0; k < n_tiles; ++k) {
        if (owner[k] < 0)
            return fail(FLP_EINVAL, "tile %lld (columns [%lld, %lld)) is held by no rank", (long long)k,
                        (long long)(k * W), (long long)((k + 1) * W < v_total ? (k + 1) * W : v_total));
        t |= (uint64_t)owner[k] << (4 * k);
    }
    *table = t;
    return FLP_OK;
}

flp_status merge_impl(const float* part_max, const float* part_sum, const float* sel, int64_t rank_stride,
                      uint64_t tile_rank, const int64_t* targets, int64_t ignore_index,
                      const uint8_t* active_mask, int64_t n, int64_t v_total, float inv_temperature, float* logp,
                      float* lse, float* lse_lo, flp_stream_t stream) {
    const void* ptrs[] = {part_max, part_sum, sel, targets, logp, lse, lse_lo, active_mask};
    const char* names[] = {"part_max", "part_sum", "sel", "targets", "logp", "lse", "lse_lo", "active_mask"};
    const bool optional[] = {false, false, false, false, false, false, true, true};
    int dev;
    flp_status st;
    if ((st = common_device(8, ptrs, names, optional, &dev)) != FLP_OK) return st;
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;

    const int64_t W = tile_width(v_total);
    const int n_tiles = (int)ceil_div(v_total, W);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rows_per_block = 256 / 16;
    flp::k_logp_merge<<<grid_for(ceil_div(n, rows_per_block)), 256, 0, s>>>(
        part_max, part_sum, sel, targets, ignore_index, active_mask, n, v_total, n_tiles, inv_temperature, logp,
        lse, lse_lo, rank_stride, tile_rank, W);
    return check_launch("merge");
}

}  // namespace

extern "C" {

flp_status fused_logp_backward_ex(const void* logits, int dtype, int64_t n, int64_t v, int64_t ld,
                                  const int64_t* targets, int64_t ignore_index,
                                  const uint8_t* active_mask, float inv_temperature,
                                  const float* lse, const float* lse_lo, const float* grad,
                                  void* dlogits, int64_t ld_out, flp_stream_t stream) {
    return backward_impl(logits, dtype, n, v, ld, 0, v, targets, ignore_index, active_mask, inv_temperature, lse,
                         lse_lo, grad, dlogits, ld_out, stream);
}

flp_status logp_shard_backward_ex(const void* shard_logits, int dtype, int64_t n, int64_t ld_shard,
                                  int64_t vocab_start, int64_t real_width, int64_t v_total,
                                  const int64_t* targets, int64_t ignore_index, const uint8_t* active_mask,
                                  float inv_temperature, const float* lse, const float* lse_lo,
                                  const float* grad, void* dshard, int64_t ld_out, flp_stream_t stream) {
    if (v_total < 1) return fail(FLP_EINVAL, "v_total must be >= 1 (got %lld)", (long long)v_total);
    if (real_width < 1) return fail(FLP_EINVAL, "real_width must be >= 1 (got %lld)", (long long)real_width);
    return backward_impl(shard_logits, dtype, n, real_width, ld_shard, vocab_start, v_total, targets,
                         ignore_index, active_mask, inv_temperature, lse, lse_lo, grad, dshard, ld_out, stream);
}

flp_status logp_shard_backward(const void* shard_logits, int64_t n, int64_t ld_shard, int64_t vocab_start,
                               int64_t real_width, int64_t v_total, const int64_t* targets, int64_t ignore_index,
                               const float* lse, const float* lse_lo, const float* grad, void* dshard,
                               int64_t ld_out, flp_stream_t stream) {
    return logp_shard_backward_ex(shard_logits, FLP_DTYPE_BF16, n, ld_shard, vocab_start, real_width, v_total,
                                  targets, ignore_index, nullptr, 1.f, lse, lse_lo, grad, dshard, ld_out, stream);
}

flp_status logp_merge_gathered_partials_ex(const float* gathered, int64_t rank_stride, int64_t world,
                                           const int64_t* vocab_starts, const int64_t* real_widths,
                                           const int64_t* targets, int64_t ignore_index,
                                           const uint8_t* active_mask, int64_t n, int64_t v_total,
                                           float inv_temperature, float* logp, float* lse, float* lse_lo,
                                           flp_stream_t stream) {
    flp_status st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v_total < 1) return fail(FLP_EINVAL, "v_total must be >= 1");
    uint64_t table = 0;
    if ((st = tile_rank_table(world, vocab_starts, real_widths, v_total, &table)) != FLP_OK) return st;
    int64_t block;
    if (__builtin_mul_overflow(n, (int64_t)(2 * flp::kTiles + 1), &block))
        return fail(FLP_EINVAL, "partials extent overflows int64");
    if (world > 1 && rank_stride < block)
        return fail(FLP_EINVAL, "rank_stride (%lld) is below one rank's %lld floats of partials",
                    (long long)rank_stride, (long long)block);
    if (world == 1) rank_stride = 0;
    if (n == 0) return ok();
    if (gathered == nullptr) return fail(FLP_EINVAL, "gathered is a null pointer");
    return merge_impl(gathered, gathered + flp::kTiles * n, gathered + 2 * flp::kTiles * n, rank_stride, table,
                      targets, ignore_index, active_mask, n, v_total, inv_temperature, logp, lse, lse_lo, stream);
}

flp_status fused_logp_backward(const void* logits, int64_t n, int64_t v, int64_t ld,
                               const int64_t* targets, int64_t ignore_index, const float* lse,
                               const float* lse_lo, const float* grad, void* dlogits,
                               int64_t ld_out, flp_stream_t stream) {
    return fused_logp_backward_ex(logits, FLP_DTYPE_BF16, n, v, ld, targets, ignore_index, nullptr,
                                  1.f, lse, lse_lo, grad, dlogits, ld_out, stream);
}

flp_status logp_shard_partials_ex(const void* shard_logits, int dtype, int64_t n, int64_t ld_shard,
                                  int64_t vocab_start, int64_t real_width, int64_t v_total,
                                  float inv_temperature, const int64_t* targets, float* part_max,
                                  float* part_sum, float* sel, flp_stream_t stream) {
    flp_status st;
    if ((st = check_dtype(dtype)) != FLP_OK) return st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v_total < 1) return fail(FLP_EINVAL, "v_total must be >= 1");
    if (real_width < 1) return fail(FLP_EINVAL, "real_width must be >= 1");
    if (vocab_start < 0 || vocab_start + real_width > v_total)
        return fail(FLP_EINVAL, "shard [%lld, %lld) is outside the vocabulary [0, %lld)",
                    (long long)vocab_start, (long long)(vocab_start + real_width), (long long)v_total);
    if (ld_shard < real_width) return fail(FLP_EINVAL, "ld_shard must be >= real_width");
    const int64_t W = tile_width(v_total);
    if (vocab_start % W != 0)
        return fail(FLP_EUNSUPPORTED, "vocab_start %lld is not a multiple of the tile width %lld",
                    (long long)vocab_start, (long long)W);
    if (vocab_start + real_width != v_total && real_width % W != 0)
        return fail(FLP_EUNSUPPORTED,
                    "real_width %lld is not a multiple of the tile width %lld and the shard "
                    "does not end the vocabulary", (long long)real_width, (long long)W);
    if (n == 0) return ok();
    int64_t bytes;
    if (!span_bytes(n, real_width, ld_shard, elem_bytes(dtype), &bytes))
        return fail(FLP_EINVAL, "shard extent overflows int64");
    const void* ptrs[] = {shard_logits, targets, part_max, part_sum, sel};
    const char* names[] = {"shard_logits", "targets", "part_max", "part_sum", "sel"};
    int dev;
    if ((st = common_device(5, ptrs, names, nullptr, &dev)) != FLP_OK) return st;
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;

    const PartArgs a{shard_logits, n, ld_shard, real_width, W, (int)(vocab_start / W),
                     (int)ceil_div(real_width, W), vocab_start, targets, make_scale(inv_temperature),
                     part_max, part_sum, sel, reinterpret_cast<cudaStream_t>(stream),
                     rows_aligned16(shard_logits, ld_shard, dtype)};
    if (dtype == FLP_DTYPE_BF16) launch_partials_d<flp::Dt::BF16>(a);
    else if (dtype == FLP_DTYPE_F16) launch_partials_d<flp::Dt::F16>(a);
    else launch_partials_d<flp::Dt::F32>(a);
    return check_launch("shard partials");
}

flp_status logp_shard_partials(const void* shard_logits, int64_t n, int64_t ld_shard,
                               int64_t vocab_start, int64_t real_width, int64_t v_total,
                               const int64_t* targets, float* part_max, float* part_sum,
                               float* sel, flp_stream_t stream) {
    return logp_shard_partials_ex(shard_logits, FLP_DTYPE_BF16, n, ld_shard, vocab_start,
                                  real_width, v_total, 1.f, targets, part_max, part_sum, sel, stream);
}

flp_status logp_merge_partials_ex(const float* part_max, const float* part_sum, const float* sel,
                                  const int64_t* targets, int64_t ignore_index,
                                  const uint8_t* active_mask, int64_t n, int64_t v_total,
                                  float inv_temperature, float* logp, float* lse, float* lse_lo,
                                  flp_stream_t stream) {
    flp_status st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v_total < 1) return fail(FLP_EINVAL, "v_total must be >= 1");
    if (n == 0) return ok();
    return merge_impl(part_max, part_sum, sel, 0, 0, targets, ignore_index, active_mask, n, v_total,
                      inv_temperature, logp, lse, lse_lo, stream);
}

flp_status logp_merge_partials(const float* part_max, const float* part_sum, const float* sel,
                               const int64_t* targets, int64_t ignore_index, int64_t n,
                               int64_t v_total, float* logp, float* lse, float* lse_lo,
                               flp_stream_t stream) {
    return logp_merge_partials_ex(part_max, part_sum, sel, targets, ignore_index, nullptr, n,
                                  v_total, 1.f, logp, lse, lse_lo, stream);
}

flp_status fused_linear_logp_workspace_size(int64_t n, int64_t v, int64_t* bytes) {
    if (bytes == nullptr) return fail(FLP_EINVAL, "bytes is a null pointer");
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v < 1) return fail(FLP_EINVAL, "v must be >= 1 (got %lld)", (long long)v);
    if (!linear_workspace_bytes(n, v, bytes)) return fail(FLP_EINVAL, "workspace size overflows int64");
    return ok();
}

flp_status fused_linear_logp_forward(const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                     const void* weight, int64_t v, int64_t ld_w, const int64_t* targets,
                                     int64_t ignore_index, const uint8_t* active_mask, float inv_temperature,
                                     void* workspace, int64_t workspace_bytes, float* logp, float* lse,
                                     float* lse_lo, flp_stream_t stream) {
    flp_status st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (d < 1) return fail(FLP_EINVAL, "d must be >= 1 (got %lld)", (long long)d);
    if (v < 1) return fail(FLP_EINVAL, "v must be >= 1 (got %lld)", (long long)v);
    if (ld_h < d || ld_w < d)
        return fail(FLP_EINVAL, "ld_h (%lld) and ld_w (%lld) must be >= d (%lld)", (long long)ld_h,
                    (long long)ld_w, (long long)d);
    if (n == 0) return ok();
    const int64_t kMaxDim = ((int64_t)1 << 31) - 1;
    if (n > kMaxDim || v > kMaxDim || d > kMaxDim)
        return fail(FLP_EUNSUPPORTED, "n, v and d must be below 2^31");
    if (!aligned16(hidden) || !aligned16(weight) || (ld_h % 8) != 0 || (ld_w % 8) != 0)
        return fail(FLP_EUNSUPPORTED,
                    "hidden and weight must start on 16-byte boundaries with row strides a multiple of 8 elements");
    int64_t bytes_h, bytes_w, need;
    if (!span_bytes(n, d, ld_h, 2, &bytes_h) || !span_bytes(v, d, ld_w, 2, &bytes_w))
        return fail(FLP_EINVAL, "hidden or weight extent overflows int64");
    if (!linear_workspace_bytes(n, v, &need)) return fail(FLP_EINVAL, "workspace size overflows int64");
    if (workspace_bytes < need)
        return fail(FLP_EINVAL, "workspace_bytes (%lld) is below the %lld bytes needed", (long long)workspace_bytes,
                    (long long)need);
    if (!aligned16(workspace)) return fail(FLP_EINVAL, "workspace must start on a 16-byte boundary");
    const void* ptrs[] = {hidden, weight, targets, workspace, logp, lse, lse_lo, active_mask};
    const char* names[] = {"hidden", "weight", "targets", "workspace", "logp", "lse", "lse_lo", "active_mask"};
    const bool optional[] = {false, false, false, false, false, false, true, true};
    int dev;
    if ((st = common_device(8, ptrs, names, optional, &dev)) != FLP_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float* ws = static_cast<float*>(workspace);
    if ((st = linear_partials_launch(dev, hidden, n, d, ld_h, weight, v, ld_w, 0, v, targets, ignore_index,
                                     active_mask, inv_temperature, ws, s)) != FLP_OK)
        return st;
    return linear_merge_launch(dev, ws, n, v, targets, ignore_index, active_mask, inv_temperature, logp, lse,
                               lse_lo, s);
}

flp_status fused_linear_logp_shard_partials(const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                            const void* weight_shard, int64_t real_width, int64_t ld_w,
                                            int64_t vocab_start, int64_t v_total, const int64_t* targets,
                                            float inv_temperature, void* workspace, int64_t workspace_bytes,
                                            flp_stream_t stream) {
    flp_status st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (d < 1) return fail(FLP_EINVAL, "d must be >= 1 (got %lld)", (long long)d);
    if (real_width < 1 || vocab_start < 0 || v_total < 1 || vocab_start + real_width > v_total)
        return fail(FLP_EINVAL, "the shard [%lld, %lld) must lie inside [0, %lld)", (long long)vocab_start,
                    (long long)(vocab_start + real_width), (long long)v_total);
    if (ld_h < d || ld_w < d) return fail(FLP_EINVAL, "ld_h and ld_w must be >= d (%lld)", (long long)d);
    if (vocab_start % flp::kLinBN != 0)
        return fail(FLP_EUNSUPPORTED, "vocab_start (%lld) must be a multiple of the %d-column tile",
                    (long long)vocab_start, flp::kLinBN);
    if (n == 0) return ok();
    const int64_t kMaxDim = ((int64_t)1 << 31) - 1;
    if (n > kMaxDim || v_total > kMaxDim || d > kMaxDim)
        return fail(FLP_EUNSUPPORTED, "n, v_total and d must be below 2^31");
    if (!aligned16(hidden) || !aligned16(weight_shard) || (ld_h % 8) != 0 || (ld_w % 8) != 0)
        return fail(FLP_EUNSUPPORTED,
                    "hidden and weight must start on 16-byte boundaries with row strides a multiple of 8 elements");
    int64_t span, need;
    if (!span_bytes(n, d, ld_h, 2, &span) || !span_bytes(real_width, d, ld_w, 2, &span))
        return fail(FLP_EINVAL, "hidden or weight extent overflows int64");
    if (!linear_workspace_bytes(n, v_total, &need)) return fail(FLP_EINVAL, "workspace size overflows int64");
    if (workspace_bytes < need)
        return fail(FLP_EINVAL, "workspace_bytes (%lld) is below the %lld bytes needed", (long long)workspace_bytes,
                    (long long)need);
    if (!aligned16(workspace)) return fail(FLP_EINVAL, "workspace must start on a 16-byte boundary");
    const void* ptrs[] = {hidden, weight_shard, targets, workspace};
    const char* names[] = {"hidden", "weight_shard", "targets", "workspace"};
    int dev;
    if ((st = common_device(4, ptrs, names, nullptr, &dev)) != FLP_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;
    // the merge decides which rows are active; every in-shard target's logit is kept
    return linear_partials_launch(dev, hidden, n, d, ld_h, weight_shard, real_width, ld_w, vocab_start, v_total,
                                  targets, -1, nullptr, inv_temperature, static_cast<float*>(workspace),
                                  reinterpret_cast<cudaStream_t>(stream));
}

flp_status fused_linear_logp_merge(const void* workspace, int64_t workspace_bytes, int64_t n, int64_t v_total,
                                   const int64_t* targets, int64_t ignore_index, const uint8_t* active_mask,
                                   float inv_temperature, float* logp, float* lse, float* lse_lo,
                                   flp_stream_t stream) {
    flp_status st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v_total < 1) return fail(FLP_EINVAL, "v_total must be >= 1 (got %lld)", (long long)v_total);
    if (n == 0) return ok();
    int64_t need;
    if (!linear_workspace_bytes(n, v_total, &need)) return fail(FLP_EINVAL, "workspace size overflows int64");
    if (workspace_bytes < need)
        return fail(FLP_EINVAL, "workspace_bytes (%lld) is below the %lld bytes needed", (long long)workspace_bytes,
                    (long long)need);
    if (!aligned16(workspace)) return fail(FLP_EINVAL, "workspace must start on a 16-byte boundary");
    const void* ptrs[] = {workspace, targets, logp, lse, lse_lo, active_mask};
    const char* names[] = {"workspace", "targets", "logp", "lse", "lse_lo", "active_mask"};
    const bool optional[] = {false, false, false, false, true, true};
    int dev;
    if ((st = common_device(6, ptrs, names, optional, &dev)) != FLP_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;
    return linear_merge_launch(dev, static_cast<const float*>(workspace), n, v_total, targets, ignore_index,
                               active_mask, inv_temperature, logp, lse, lse_lo,
                               reinterpret_cast<cudaStream_t>(stream));
}

flp_status fused_linear_logp_merge_gathered(const float* gathered, int64_t rank_stride, int world,
                                            const int64_t* vocab_starts, const int64_t* real_widths, int64_t n,
                                            int64_t v_total, const int64_t* targets, int64_t ignore_index,
                                            const uint8_t* active_mask, float inv_temperature, float* logp,
                                            float* lse, float* lse_lo, flp_stream_t stream) {
    flp_status st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v_total < 1) return fail(FLP_EINVAL, "v_total must be >= 1 (got %lld)", (long long)v_total);
    if (world < 1 || world > flp::kLinMaxRanks)
        return fail(FLP_EINVAL, "world must be in [1, %d] (got %d)", flp::kLinMaxRanks, world);
    if (vocab_starts == nullptr || real_widths == nullptr)
        return fail(FLP_EINVAL, "vocab_starts and real_widths are host arrays of world entries");
    const int64_t nvt = linear_vocab_tiles(v_total);
    if (nvt > INT32_MAX) return fail(FLP_EINVAL, "too many vocabulary tiles");
    int64_t need;   // floats of one rank's block: tile maxima and sums [n, nvt] each, selected logits [n]
    if (__builtin_mul_overflow(2 * nvt + 1, n, &need)) return fail(FLP_EINVAL, "block size overflows int64");
    if (rank_stride < need)
        return fail(FLP_EINVAL, "rank_stride (%lld floats) is below one rank's block (%lld floats)",
                    (long long)rank_stride, (long long)need);
    // each rank's tiles, on the 256-column grid, covering every tile once
    flp::LinRankTiles rt;
    rt.world = world;
    int order[flp::kLinMaxRanks];
    for (int r = 0; r < world; ++r) {
        const int64_t a = vocab_starts[r], w = real_widths[r];
        if (w < 1 || a < 0 || a > v_total - w)
            return fail(FLP_EINVAL, "rank %d: columns [%lld, %lld) are not inside the vocabulary [0, %lld)", r,
                        (long long)a, (long long)(a + w), (long long)v_total);
        if (a % flp::kLinBN != 0 || (a + w != v_total && w % flp::kLinBN != 0))
            return fail(FLP_EUNSUPPORTED, "rank %d: columns [%lld, %lld) are off the %d-column tile grid", r,
                        (long long)a, (long long)(a + w), flp::kLinBN);
        order[r] = r;
    }
    for (int i = 1; i < world; ++i)   // by first column (insertion sort, at most 16)
        for (int j = i; j > 0 && vocab_starts[order[j]] < vocab_starts[order[j - 1]]; --j) {
            const int tmp = order[j];
            order[j] = order[j - 1];
            order[j - 1] = tmp;
        }
    int64_t next = 0;
    for (int j = 0; j < world; ++j) {
        const int r = order[j];
        const int64_t t0 = vocab_starts[r] / flp::kLinBN, t1 = ceil_div(vocab_starts[r] + real_widths[r], flp::kLinBN);
        if (t0 != next)
            return fail(FLP_EINVAL, "tile %lld (columns from %lld) is %s", (long long)next,
                        (long long)(next * flp::kLinBN), t0 > next ? "held by no rank" : "held by two ranks");
        rt.t0[j] = (int)t0;
        rt.t1[j] = (int)t1;
        rt.rank[j] = r;
        next = t1;
    }
    if (next != nvt)
        return fail(FLP_EINVAL, "tiles from %lld (columns from %lld) are held by no rank", (long long)next,
                    (long long)(next * flp::kLinBN));
    for (int j = world; j < flp::kLinMaxRanks; ++j) rt.t0[j] = rt.t1[j] = rt.rank[j] = 0;
    if (n == 0) return ok();
    const void* ptrs[] = {gathered, targets, logp, lse, lse_lo, active_mask};
    const char* names[] = {"gathered", "targets", "logp", "lse", "lse_lo", "active_mask"};
    const bool optional[] = {false, false, false, false, true, true};
    int dev;
    if ((st = common_device(6, ptrs, names, optional, &dev)) != FLP_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;
    const int sms = sm_count(dev);
    if (sms <= 0) return fail(FLP_ECUDA, "cannot read the SM count of device %d", dev);
    const int64_t ctas = ceil_div(n * 32, flp::kLinMergeThreads);
    flp::k_linear_logp_merge_gathered<<<(int)(ctas < (int64_t)sms * 16 ? ctas : (int64_t)sms * 16),
                                        flp::kLinMergeThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        gathered, rank_stride, rt, n, (int)nvt, v_total, targets, ignore_index, active_mask, inv_temperature, logp,
        lse, lse_lo);
    return check_launch("linear logp gathered merge");
}

flp_status flp_sum_blocks(const float* blocks, int64_t block_stride, int world, int64_t rows, int64_t cols,
                          float* out, int64_t ld_out, flp_stream_t stream) {
    flp_status st;
    if (world < 1) return fail(FLP_EINVAL, "world must be >= 1 (got %d)", world);
    if (rows < 0 || cols < 0) return fail(FLP_EINVAL, "rows and cols must be >= 0");
    if (ld_out < cols) return fail(FLP_EINVAL, "ld_out (%lld) must be >= cols (%lld)", (long long)ld_out,
                                   (long long)cols);
    int64_t total;
    if (__builtin_mul_overflow(rows, cols, &total)) return fail(FLP_EINVAL, "rows * cols overflows int64");
    if (world > 1 && block_stride < total)
        return fail(FLP_EINVAL, "block_stride (%lld) is below one block (%lld floats)", (long long)block_stride,
                    (long long)total);
    if (total == 0) return ok();
    const void* ptrs[] = {blocks, out};
    const char* names[] = {"blocks", "out"};
    const bool optional[] = {false, false};
    int dev;
    if ((st = common_device(2, ptrs, names, optional, &dev)) != FLP_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;
    const int sms = sm_count(dev);
    if (sms <= 0) return fail(FLP_ECUDA, "cannot read the SM count of device %d", dev);
    const int64_t blocks_n = ceil_div(total, 256);
    flp::k_sum_blocks_ordered<<<(int)(blocks_n < (int64_t)sms * 8 ? blocks_n : (int64_t)sms * 8), 256, 0,
                                reinterpret_cast<cudaStream_t>(stream)>>>(blocks, block_stride, world, rows, cols,
                                                                           out, ld_out);
    return check_launch("ordered block sum");
}

flp_status fused_linear_logp_backward_workspace_size(int64_t d, int64_t v, int64_t* bytes) {
    if (bytes == nullptr) return fail(FLP_EINVAL, "bytes is a null pointer");
    if (d < 1 || v < 1) return fail(FLP_EINVAL, "d and v must be >= 1");
    int64_t ld, off_dh;
    if (!linear_grad_workspace(d, v, &ld, &off_dh, bytes))
        return fail(FLP_EINVAL, "workspace size overflows int64");
    return ok();
}

}  // extern "C"

namespace {

// The backward for weight rows = global vocabulary columns [vocab_start,
// vocab_start + v) of a v_total-column vocabulary (the whole head: 0, v).
flp_status linear_backward_impl(const void* hidden, int64_t n, int64_t d, int64_t ld_h, const void* weight,
                                int64_t v, int64_t ld_w, int64_t vocab_start, int64_t v_total,
                                const int64_t* targets, int64_t ignore_index, const uint8_t* active_mask,
                                float inv_temperature, const float* lse, const float* lse_lo, const float* grad,
                                void* workspace, int64_t workspace_bytes, float* dhidden, int64_t ld_dh,
                                int accumulate_dhidden, float* dweight, int64_t ld_dw, int accumulate_dweight,
                                flp_stream_t stream) {
    flp_status st;
    if ((st = check_scale(inv_temperature)) != FLP_OK) return st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (d < 1) return fail(FLP_EINVAL, "d must be >= 1 (got %lld)", (long long)d);
    if (v < 1) return fail(FLP_EINVAL, "v must be >= 1 (got %lld)", (long long)v);
    if (ld_h < d || ld_w < d || ld_dh < d || ld_dw < d)
        return fail(FLP_EINVAL, "ld_h, ld_w, ld_dh and ld_dw must be >= d (%lld)", (long long)d);
    const int64_t kMaxDim = ((int64_t)1 << 31) - 1;
    if (n > kMaxDim || v > kMaxDim || d > kMaxDim || ld_w > kMaxDim || ld_h > kMaxDim || ld_dh > kMaxDim ||
        ld_dw > kMaxDim)
        return fail(FLP_EUNSUPPORTED, "sizes and strides must be below 2^31");
    if (!aligned16(hidden) || !aligned16(weight) || (ld_h % 8) != 0 || (ld_w % 8) != 0)
        return fail(FLP_EUNSUPPORTED,
                    "hidden and weight must start on 16-byte boundaries with row strides a multiple of 8 elements");
    int64_t span;
    if (!span_bytes(v, d, ld_w, 2, &span) || !span_bytes(v, d, ld_dw, 4, &span) ||
        (n > 0 && (!span_bytes(n, d, ld_h, 2, &span) || !span_bytes(n, d, ld_dh, 4, &span))))
        return fail(FLP_EINVAL, "an operand's extent overflows int64");
    if (vocab_start < 0 || vocab_start + v > v_total)
        return fail(FLP_EINVAL, "the weight rows [%lld, %lld) must lie inside [0, %lld)", (long long)vocab_start,
                    (long long)(vocab_start + v), (long long)v_total);
    if (vocab_start % flp::kLinBN != 0)
        return fail(FLP_EUNSUPPORTED, "vocab_start (%lld) must be a multiple of the %d-column tile",
                    (long long)vocab_start, flp::kLinBN);
    if (n == 0 && accumulate_dweight) return ok();   // no rows add nothing
    if (n == 0) {   // no rows: dW = 0, nothing else is read
        int dev0;
        if ((st = device_of(dweight, "dweight", &dev0)) != FLP_OK) return st;
        DeviceGuard g0;
        if ((st = g0.enter(dev0)) != FLP_OK) return st;
        const cudaError_t e = cudaMemset2DAsync(dweight, (size_t)ld_dw * 4, 0, (size_t)d * 4, (size_t)v,
                                                reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return fail(FLP_ECUDA, "clearing dweight: %s", cudaGetErrorString(e));
        return ok();
    }
    int64_t ld_dz, off_dh, need;
    if (!linear_grad_workspace(d, v, &ld_dz, &off_dh, &need))
        return fail(FLP_EINVAL, "workspace size overflows int64");
    if (workspace_bytes < need)
        return fail(FLP_EINVAL, "workspace_bytes (%lld) is below the %lld bytes needed", (long long)workspace_bytes,
                    (long long)need);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(FLP_EINVAL, "workspace must start on a 256-byte boundary");
    const void* ptrs[] = {hidden, weight, targets, lse, grad, workspace, dhidden, dweight, lse_lo, active_mask};
    const char* names[] = {"hidden", "weight", "targets", "lse", "grad", "workspace", "dhidden", "dweight",
                           "lse_lo", "active_mask"};
    const bool optional[] = {false, false, false, false, false, false, false, false, true, true};
    int dev;
    if ((st = common_device(10, ptrs, names, optional, &dev)) != FLP_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = linear_setup(dev)) != FLP_OK) return st;
    if ((st = gemm_setup(dev)) != FLP_OK) return st;
    const int sms = sm_count(dev);
    if (sms <= 0) return fail(FLP_ECUDA, "cannot read the SM count of device %d", dev);

    // the weight as the dZ kernel's K-major operand and as dH's MN-major B
    CUtensorMap tm_w, tm_w_mn;
    if ((st = make_tmap_bf16(&tm_w, weight, v, d, ld_w, flp::kLinBN, "weight")) != FLP_OK) return st;
    if ((st = make_tmap_bf16(&tm_w_mn, weight, v, d, ld_w, 64, "weight")) != FLP_OK) return st;
    char* ws = static_cast<char*>(workspace);
    uint16_t* dz = reinterpret_cast<uint16_t*>(ws);
    float* dh_parts = reinterpret_cast<float*>(ws + off_dh);
    const int splits = dh_splits(v);
    const int64_t nvt = linear_vocab_tiles(v);
    const char* hb = static_cast<const char*>(hidden);
    for (int64_t start = 0; start < n; start += kLinGradChunk) {
        const int64_t rows = (n - start < kLinGradChunk) ? n - start : kLinGradChunk;
        const void* h_chunk = hb + start * ld_h * 2;
        // dZ of the chunk's rows, in BF16, recomputed on the tensor cores
        CUtensorMap tm_h, tm_h_mn, tm_dz, tm_dz_mn;
        if ((st = make_tmap_bf16(&tm_h, h_chunk, rows, d, ld_h, flp::kLinBM, "hidden")) != FLP_OK) return st;
        if ((st = make_tmap_bf16(&tm_h_mn, h_chunk, rows, d, ld_h, 64, "hidden")) != FLP_OK) return st;
        if ((st = make_tmap_bf16(&tm_dz, dz, rows, v, ld_dz, flp::kGemmBM, "dZ")) != FLP_OK) return st;
        if ((st = make_tmap_bf16(&tm_dz_mn, dz, rows, v, ld_dz, 64, "dZ")) != FLP_OK) return st;
        const int64_t nrb = ceil_div(rows, flp::kLinBM);
        const int64_t ntiles = nrb * nvt;
        flp::LinArgs a;
        a.n = rows;
        a.v = v;
        a.nrb = (int)nrb;
        a.nvt = (int)nvt;
        a.nkb = (int)ceil_div(d, flp::kLinBK);
        a.vocab_start = vocab_start;
        a.v_total = v_total;
        a.vt0 = (int)(vocab_start / flp::kLinBN);
        a.nvt_total = (int)linear_vocab_tiles(v_total);
        a.y = targets + start;
        a.ignore_index = ignore_index;
        a.mask = active_mask ? active_mask + start : nullptr;
        a.sc = make_scale(inv_temperature);
        a.pm = a.ps = a.xsel = nullptr;
        a.n_valid = rows;
        a.lse = lse + start;
        a.lse_lo = lse_lo ? lse_lo + start : nullptr;
        a.g = grad + start;
        a.inv_s = 1.f / inv_temperature;
        a.dz = dz;
        a.ld_dz = ld_dz;
        flp::k_linear_logp_tiles<true><<<(int)(ntiles < sms ? ntiles : sms), flp::kLinThreads, flp::kLinSmemBytes,
                                          s>>>(tm_h, tm_w, a);
        if ((st = check_launch("linear logp gradient tiles")) != FLP_OK) return st;
        // dH rows = dZ W (K = the vocabulary), in fixed K splits summed in split order
        float* dh_rows = dhidden + start * ld_dh;
        if (splits == 1) {
            if ((st = gemm_launch<false>(dev, sms, tm_dz, tm_w_mn, rows, d, v, 1, dh_rows, ld_dh, 0, rows,
                                         accumulate_dhidden != 0, s, "dhidden product")) != FLP_OK)
                return st;
        } else {
            const int64_t stride = kLinGradChunk * d;
            if ((st = gemm_launch<false>(dev, sms, tm_dz, tm_w_mn, rows, d, v, splits, dh_parts, d, stride, 0, false,
                                         s, "dhidden product")) != FLP_OK)
                return st;
            const int64_t blocks = ceil_div(rows * d, 256);
            flp::k_gemm_split_sum<<<(int)(blocks < (int64_t)sms * 8 ? blocks : (int64_t)sms * 8), 256, 0, s>>>(
                dh_parts, splits, stride, d, rows, d, dh_rows, ld_dh, accumulate_dhidden);
            if ((st = check_launch("dhidden split sum")) != FLP_OK) return st;
        }
        // dW (+)= dZ^T H (K = the chunk's rows), added chunk after chunk in row order
        if ((st = gemm_launch<true>(dev, sms, tm_dz_mn, tm_h_mn, v, d, rows, 1, dweight, ld_dw, 0, v,
                                    start > 0 || accumulate_dweight, s, "dweight product")) != FLP_OK)
            return st;
    }
    return ok();
}

}  // namespace

extern "C" {

flp_status fused_linear_logp_backward(const void* hidden, int64_t n, int64_t d, int64_t ld_h, const void* weight,
                                      int64_t v, int64_t ld_w, const int64_t* targets, int64_t ignore_index,
                                      const uint8_t* active_mask, float inv_temperature, const float* lse,
                                      const float* lse_lo, const float* grad, void* workspace,
                                      int64_t workspace_bytes, float* dhidden, int64_t ld_dh, float* dweight,
                                      int64_t ld_dw, int accumulate_dweight, flp_stream_t stream) {
    return linear_backward_impl(hidden, n, d, ld_h, weight, v, ld_w, 0, v, targets, ignore_index, active_mask,
                                inv_temperature, lse, lse_lo, grad, workspace, workspace_bytes, dhidden, ld_dh, 0,
                                dweight, ld_dw, accumulate_dweight, stream);
}

flp_status fused_linear_logp_shard_backward(const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                            const void* weight_shard, int64_t real_width, int64_t ld_w,
                                            int64_t vocab_start, int64_t v_total, const int64_t* targets,
                                            int64_t ignore_index, const uint8_t* active_mask, float inv_temperature,
                                            const float* lse, const float* lse_lo, const float* grad,
                                            void* workspace, int64_t workspace_bytes, float* dhidden,
                                            int64_t ld_dh, int accumulate_dhidden, float* dweight_shard,
                                            int64_t ld_dw, int accumulate_dweight, flp_stream_t stream) {
    if (real_width < 1) return fail(FLP_EINVAL, "real_width must be >= 1 (got %lld)", (long long)real_width);
    return linear_backward_impl(hidden, n, d, ld_h, weight_shard, real_width, ld_w, vocab_start, v_total, targets,
                                ignore_index, active_mask, inv_temperature, lse, lse_lo, grad, workspace,
                                workspace_bytes, dhidden, ld_dh, accumulate_dhidden, dweight_shard, ld_dw,
                                accumulate_dweight, stream);
}

flp_status fused_linear_logp_forward_noalloc(const void* hidden, int64_t n, int64_t d, int64_t ld_h,
                                             const void* weight, int64_t v, int64_t ld_w,
                                             const int64_t* targets, int64_t ignore_index,
                                             const uint8_t* active_mask, float inv_temperature, float* logp,
                                             float* lse, float* lse_lo, flp_stream_t stream) {
    // empty or malformed sizes: the same answers as the workspace entry point
    if (n <= 0 || v < 1 || d < 1)
        return fused_linear_logp_forward(hidden, n, d, ld_h, weight, v, ld_w, targets, ignore_index, active_mask,
                                         inv_temperature, nullptr, 0, logp, lse, lse_lo, stream);
    int64_t need;
    if (!linear_workspace_bytes(n, v, &need)) return fail(FLP_EINVAL, "scratch size overflows int64");
    if (need > kNoAllocScratchBytes)
        return fail(FLP_EUNSUPPORTED,
                    "fused_linear_logp_forward_noalloc: %lld rows with a %lld-entry vocabulary need %lld bytes of "
                    "scratch, more than its fixed %lld bytes; pass fewer rows per call or use "
                    "fused_linear_logp_forward with a workspace",
                    (long long)n, (long long)v, (long long)need, (long long)kNoAllocScratchBytes);
    flp_status st;
    int dev;
    if ((st = device_of(hidden, "hidden", &dev)) != FLP_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    void* scratch = nullptr;
    {
        DeviceGuard guard;
        if ((st = guard.enter(dev)) != FLP_OK) return st;
        if ((st = noalloc_scratch_address(dev, &scratch)) != FLP_OK) return st;
    }
    return fused_linear_logp_forward(hidden, n, d, ld_h, weight, v, ld_w, targets, ignore_index, active_mask,
                                     inv_temperature, scratch, kNoAllocScratchBytes, logp, lse, lse_lo, stream);
}

flp_status logp_grpo_loss_workspace_size(int64_t n, int64_t num_seqs, int64_t* bytes) {
    if (bytes == nullptr) return fail(FLP_EINVAL, "bytes is a null pointer");
    if (n < 0 || num_seqs < 0) return fail(FLP_EINVAL, "n and num_seqs must be >= 0");
    *bytes = grpo_workspace_bytes(n, num_seqs);
    return ok();
}

// What a GRPO call runs: everything, only the counts, or only the token pass
// on counts that an earlier call left in the workspace.
enum GrpoStage { kGrpoWhole = 0, kGrpoCountsOnly = 1, kGrpoCounted = 2 };

// FNV-1a over the fields that fix the counts: a call that reuses counts
// must describe the same layout.
static uint64_t grpo_tag(int64_t n, int64_t nseq, int mode, float normalizer, const void* mask, const void* cu) {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&](const void* p, size_t len) {
        const unsigned char* b = static_cast<const unsigned char*>(p);
        for (size_t i = 0; i < len; ++i) h = (h ^ b[i]) * 1099511628211ull;
    };
    const uintptr_t m = reinterpret_cast<uintptr_t>(mask), c = reinterpret_cast<uintptr_t>(cu);
    mix(&n, sizeof n);
    mix(&nseq, sizeof nseq);
    mix(&mode, sizeof mode);
    mix(&normalizer, sizeof normalizer);
    mix(&m, sizeof m);
    mix(&c, sizeof c);
    return h;
}

static flp_status grpo_impl(GrpoStage stage, const float* logp, const float* old_logp, const float* ref_logp,
                            const float* advantages, const uint8_t* active_mask, const int64_t* cu_seqlens,
                            int64_t num_seqs, int64_t n, int mode, float eps_lo, float eps_hi, float beta,
                            float normalizer, void* workspace, int64_t workspace_bytes, float* loss, float* grad,
                            float* token_loss, flp_stream_t stream) {
    flp_status st;
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (mode < FLP_GRPO_TOKEN_MEAN || mode > FLP_GRPO_SEQ_MEAN_TOKEN_SUM)
        return fail(FLP_EINVAL, "mode must be 0, 1 or 2 (got %d)", mode);
    if (stage != kGrpoCountsOnly && (!(eps_lo >= 0.f && eps_lo < 1.f) || !(eps_hi >= 0.f) || !isfinite(eps_hi)))
        return fail(FLP_EINVAL, "clip range needs 0 <= eps_lo < 1 and finite eps_hi >= 0");
    if (!isfinite(beta) || !isfinite(normalizer) || normalizer < 0.f)
        return fail(FLP_EINVAL, "beta and normalizer must be finite, normalizer >= 0");
    if (cu_seqlens && (num_seqs < 0 || num_seqs >= INT32_MAX))
        return fail(FLP_EINVAL, "num_seqs must be in [0, 2^31 - 1)");
    if (!cu_seqlens && mode != FLP_GRPO_TOKEN_MEAN && num_seqs != 0 && num_seqs != 1)
        return fail(FLP_EINVAL, "sequence normalisers need cu_seqlens (or the whole batch as one sequence)");
    const int64_t nseq = cu_seqlens ? num_seqs : 0;
    const int64_t need = grpo_workspace_bytes(n, nseq);
    if (workspace_bytes < need)
        return fail(FLP_EINVAL, "workspace_bytes (%lld) is below the %lld bytes needed", (long long)workspace_bytes,
                    (long long)need);
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
        return fail(FLP_EINVAL, "workspace must start on a 16-byte boundary");
    int dev;
    if (stage == kGrpoCountsOnly) {
        const void* ptrs[] = {workspace, active_mask, cu_seqlens};
        const char* names[] = {"workspace", "active_mask", "cu_seqlens"};
        const bool optional[] = {false, true, true};
        if ((st = common_device(n == 0 ? 1 : 3, ptrs, names, optional, &dev)) != FLP_OK) return st;
    } else {
        const void* ptrs[] = {loss, workspace, logp, old_logp, advantages, grad, ref_logp, active_mask, cu_seqlens,
                              token_loss};
        const char* names[] = {"loss", "workspace", "logp", "old_logp", "advantages", "grad", "ref_logp",
                               "active_mask", "cu_seqlens", "token_loss"};
        const bool optional[] = {false, false, false, false, false, false, true, true, true, true};
        // with n == 0 only the loss (and the workspace's count words) are written
        if ((st = common_device(n == 0 ? 2 : 10, ptrs, names, optional, &dev)) != FLP_OK) return st;
    }
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;
    // with a caller's normaliser the token mean and the sequence mean of sums
    // have one weight known now: the token pass applies it and nothing is counted
    const float prescale =
        (normalizer > 0.f && mode != FLP_GRPO_SEQ_MEAN_TOKEN_MEAN) ? (float)(1.0 / (double)normalizer) : 0.f;
    // counts from an earlier call are used only when a weight depends on them
    const bool reuse = stage == kGrpoCounted && prescale == 0.f;
    const flp::GrpoArgs a{logp, old_logp, ref_logp, advantages, active_mask, cu_seqlens, nseq, n, mode,
                          eps_lo, eps_hi, beta, normalizer, prescale, loss, grad, token_loss,
                          grpo_tag(n, nseq, mode, normalizer, active_mask, cu_seqlens), reuse ? 1 : 0};
    const int64_t nchunks = ceil_div(n, flp::kGrpoChunk);
    char* base = static_cast<char*>(workspace);
    flp::GrpoWork wk;
    wk.dcnt = reinterpret_cast<int64_t*>(base);
    wk.ticket = reinterpret_cast<unsigned*>(base + 8);
    wk.tag = reinterpret_cast<uint64_t*>(base + 16);
    wk.part_t = reinterpret_cast<flp::FF*>(base + 32);
    wk.part_q = wk.part_t + flp::kGrpoPassCtas;
    wk.a_part = reinterpret_cast<int64_t*>(wk.part_q + flp::kGrpoPassCtas);
    wk.range_cnt = wk.a_part + flp::kGrpoFixMaxCtas;
    wk.seg_cnt = reinterpret_cast<float2*>(wk.range_cnt + flp::kGrpoCountMaxCtas);
    wk.word_pre = reinterpret_cast<uint32_t*>(wk.seg_cnt + nseq);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto al = [](const void* q, uintptr_t m) { return (reinterpret_cast<uintptr_t>(q) & (m - 1)) == 0; };
    int64_t nfix = (cu_seqlens != nullptr && n > 0 && mode != FLP_GRPO_TOKEN_MEAN)
                       ? ceil_div(nseq, flp::kGrpoFixThreads) : 1;
    nfix = nfix < 1 ? 1 : (nfix > flp::kGrpoFixMaxCtas ? flp::kGrpoFixMaxCtas : nfix);
    if (!reuse) {
        // 1. the mask's counts, when a weight depends on them (any weight but
        //    the caller's uniform one); ranges of R tokens (a multiple of 16),
        //    at most 1024 of them, a function of n only
        int64_t range = 0;
        int nranges = 0;
        if (n > 0 && prescale == 0.f && active_mask != nullptr) {
            int64_t g = ceil_div(n, flp::kGrpoCountRound);
            g = g < 1 ? 1 : (g > flp::kGrpoCountMaxCtas ? flp::kGrpoCountMaxCtas : g);
            range = ceil_div(ceil_div(n, g), 16) * 16;
            nranges = (int)ceil_div(n, range);
            if (al(active_mask, 16))
                flp::k_grpo_count<true><<<nranges, flp::kGrpoCountThreads, 0, s>>>(a, wk, range);
            else
                flp::k_grpo_count<false><<<nranges, flp::kGrpoCountThreads, 0, s>>>(a, wk, range);
            if ((st = check_launch("grpo count")) != FLP_OK) return st;
        }
        // 2. the sequences' counts (a sequence per thread); it waits for the
        //    count on the device when that ran before it
        auto fix = al(active_mask, 16) ? flp::k_grpo_fix<true> : flp::k_grpo_fix<false>;
        if (nranges > 0) {
            if ((st = launch_dependent("grpo counts", fix, (int)nfix, flp::kGrpoFixThreads, s, a, wk, range,
                                       nranges)) != FLP_OK)
                return st;
        } else {
            fix<<<(int)nfix, flp::kGrpoFixThreads, 0, s>>>(a, wk, range, nranges);
            if ((st = check_launch("grpo counts")) != FLP_OK) return st;
        }
    }
    if (stage == kGrpoCountsOnly) return ok();
    // 3. the token pass (launched while the fix kernel runs, when it ran in
    //    this call): final gradients and the loss; its grid is fixed by n (the
    //    fold's shape depends on it)
    if (n > 0) {
        const bool vec = al(logp, 16) && al(old_logp, 16) && al(advantages, 16) && al(grad, 16) &&
                         al(ref_logp, 16) && al(token_loss, 16) && al(active_mask, 4);
        int64_t grid = ceil_div(nchunks, flp::kGrpoPassThreads / 32);
        grid = grid < 1 ? 1 : (grid > flp::kGrpoPassCtas ? flp::kGrpoPassCtas : grid);
        const bool per_seq = cu_seqlens != nullptr && mode == FLP_GRPO_SEQ_MEAN_TOKEN_MEAN;
        auto kern = vec ? (per_seq ? flp::k_grpo_pass<true, true> : flp::k_grpo_pass<true, false>)
                        : (per_seq ? flp::k_grpo_pass<false, true> : flp::k_grpo_pass<false, false>);
        if (reuse) {
            kern<<<(int)grid, flp::kGrpoPassThreads, 0, s>>>(a, wk, (int)nfix);
            if ((st = check_launch("grpo pass")) != FLP_OK) return st;
        } else if ((st = launch_dependent("grpo pass", kern, (int)grid, flp::kGrpoPassThreads, s, a, wk,
                                          (int)nfix)) != FLP_OK) {
            return st;
        }
    } else if (reuse) {
        // no tokens: the loss is 0 and nothing else is written
        if (cudaMemsetAsync(loss, 0, sizeof(float), s) != cudaSuccess)
            return fail(FLP_ECUDA, "grpo loss: %s", cudaGetErrorString(cudaGetLastError()));
    }
    return ok();
}

flp_status logp_grpo_loss(const float* logp, const float* old_logp, const float* ref_logp,
                          const float* advantages, const uint8_t* active_mask,
                          const int64_t* cu_seqlens, int64_t num_seqs, int64_t n, int mode,
                          float eps_lo, float eps_hi, float beta, float normalizer, void* workspace,
                          int64_t workspace_bytes, float* loss, float* grad, float* token_loss,
                          flp_stream_t stream) {
    return grpo_impl(kGrpoWhole, logp, old_logp, ref_logp, advantages, active_mask, cu_seqlens, num_seqs, n, mode,
                     eps_lo, eps_hi, beta, normalizer, workspace, workspace_bytes, loss, grad, token_loss, stream);
}

flp_status logp_grpo_loss_counts(const uint8_t* active_mask, const int64_t* cu_seqlens, int64_t num_seqs,
                                 int64_t n, int mode, float normalizer, void* workspace, int64_t workspace_bytes,
                                 flp_stream_t stream) {
    return grpo_impl(kGrpoCountsOnly, nullptr, nullptr, nullptr, nullptr, active_mask, cu_seqlens, num_seqs, n, mode,
                     0.f, 0.f, 0.f, normalizer, workspace, workspace_bytes, nullptr, nullptr, nullptr, stream);
}

flp_status logp_grpo_loss_counted(const float* logp, const float* old_logp, const float* ref_logp,
                                  const float* advantages, const uint8_t* active_mask,
                                  const int64_t* cu_seqlens, int64_t num_seqs, int64_t n, int mode,
                                  float eps_lo, float eps_hi, float beta, float normalizer, void* workspace,
                                  int64_t workspace_bytes, float* loss, float* grad, float* token_loss,
                                  flp_stream_t stream) {
    return grpo_impl(kGrpoCounted, logp, old_logp, ref_logp, advantages, active_mask, cu_seqlens, num_seqs, n, mode,
                     eps_lo, eps_hi, beta, normalizer, workspace, workspace_bytes, loss, grad, token_loss, stream);
}

flp_status flp_device_error(int device, int* code) {
    if (code == nullptr) return fail(FLP_EINVAL, "code is a null pointer");
    DeviceGuard guard;
    flp_status st = guard.enter(device);
    if (st != FLP_OK) return st;
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, flp::g_device_error, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(flp::g_device_error, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(FLP_ECUDA, "device error word: %s", cudaGetErrorString(e));
    *code = v;
    return ok();
}

flp_status flp_selftest_ex2_bias(int device, double* mean_rel_err, double* compensation) {
    if (mean_rel_err == nullptr || compensation == nullptr)
        return fail(FLP_EINVAL, "output pointers must not be null");
    DeviceGuard guard;
    flp_status st = guard.enter(device);
    if (st != FLP_OK) return st;
    flp::k_ex2_bias_selftest<<<1, 1024>>>();
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    double v = 0.0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, flp::g_ex2_bias, sizeof v);
    if (e != cudaSuccess) return fail(FLP_ECUDA, "self-test: %s", cudaGetErrorString(e));
    *mean_rel_err = v;
    *compensation = (double)flp::kEx2BiasComp;
    return ok();
}

flp_status flp_selftest_wait_timeout(int device, int64_t limit_cycles, int* timed_out) {
    if (timed_out == nullptr) return fail(FLP_EINVAL, "timed_out is a null pointer");
    if (limit_cycles < 0 || limit_cycles > 100000000)
        return fail(FLP_EINVAL, "limit_cycles must be in [0, 1e8]");
    DeviceGuard guard;
    flp_status st = guard.enter(device);
    if (st != FLP_OK) return st;
    flp::k_wait_timeout_selftest<<<1, 1>>>((long long)limit_cycles);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int v = -1;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, flp::g_selftest_result, sizeof v);
    if (e != cudaSuccess) return fail(FLP_ECUDA, "self-test: %s", cudaGetErrorString(e));
    *timed_out = v;
    return ok();
}

}  // extern "C"
