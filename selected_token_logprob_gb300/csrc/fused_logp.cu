// Host side of libfused_logp.so: argument checks, device guard, launch
// configuration and the extern "C" entry points declared in
// include/fused_logp.h.  All checks run on the host before any launch and
// report through the return code (no device-side traps).
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "fused_logp.h"
#include "logp_kernels.cuh"

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
        return fail(FLP_EINVAL, "%s: cudaPointerGetAttributes failed (%s)", name,
                    cudaGetErrorString(e));
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
        return fail(FLP_EINVAL, "%s must point to device memory", name);
    *dev = a.device;
    return FLP_OK;
}

// All pointers must be device memory of one device; returns that device.
flp_status common_device(int count, const void* const* ptrs, const char* const* names,
                         int* dev) {
    int d0 = -1;
    for (int i = 0; i < count; ++i) {
        int d;
        const flp_status st = device_of(ptrs[i], names[i], &d);
        if (st != FLP_OK) return st;
        if (i == 0) d0 = d;
        else if (d != d0)
            return fail(FLP_EINVAL, "%s is on device %d but %s is on device %d", names[i], d,
                        names[0], d0);
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

constexpr int64_t kMaxGrid = 2147483647;
constexpr int kMaxDevices = 64;

// Once per device: allow the bulk-copy forward its dynamic shared memory, and
// cache the SM count used to size its persistent grid.
flp_status bulk_forward_setup(int dev, int* sms) {
    static int sm_count[kMaxDevices];
    static bool ready[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return fail(FLP_ECUDA, "device index %d out of range", dev);
    if (!ready[dev]) {
        cudaError_t e = cudaFuncSetAttribute(flp::k_logp_fwd_bulk,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             flp::kFwdSmemBytes);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(FLP_ECUDA, "forward setup: %s", cudaGetErrorString(e));
        ready[dev] = true;
    }
    *sms = sm_count[dev];
    return FLP_OK;
}

int grid_for(int64_t items) { return (int)(items < kMaxGrid ? items : kMaxGrid); }

}  // namespace

extern "C" {

const char* flp_last_error(void) { return g_msg; }

const char* flp_version(void) { return "fused_logp 0.1 (sm_103a)"; }

int64_t flp_tile_width(int64_t v) { return tile_width(v); }

flp_status fused_logp_forward(const void* logits, int64_t n, int64_t v, int64_t ld,
                              const int64_t* targets, int64_t ignore_index, float* logp,
                              float* lse, float* lse_lo, flp_stream_t stream) {
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v < 1) return fail(FLP_EINVAL, "v must be >= 1 (got %lld)", (long long)v);
    if (ld < v) return fail(FLP_EINVAL, "ld (%lld) must be >= v (%lld)", (long long)ld, (long long)v);
    if (n == 0) return ok();
    int64_t bytes;
    if (!span_bytes(n, v, ld, 2, &bytes)) return fail(FLP_EINVAL, "logits extent overflows int64");
    const void* ptrs[] = {logits, targets, logp, lse, lse_lo ? lse_lo : lse};
    const char* names[] = {"logits", "targets", "logp", "lse", "lse_lo"};
    int dev;
    flp_status st = common_device(5, ptrs, names, &dev);
    if (st != FLP_OK) return st;
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;

    const int64_t W = tile_width(v);
    const uint16_t* x = static_cast<const uint16_t*>(logits);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (aligned16(x) && ld % 8 == 0 && v < ((int64_t)1 << 31)) {
        int sms;
        if ((st = bulk_forward_setup(dev, &sms)) != FLP_OK) return st;
        const int grid = grid_for(n < 2 * (int64_t)sms ? n : 2 * (int64_t)sms);
        flp::k_logp_fwd_bulk<<<grid, flp::kFwdThreads, flp::kFwdSmemBytes, s>>>(
            x, n, v, ld, W, targets, ignore_index, logp, lse, lse_lo);
    } else {
        flp::k_logp_fwd<false><<<grid_for(n), flp::kFwdThreads, 0, s>>>(
            x, n, v, ld, W, targets, ignore_index, logp, lse, lse_lo);
    }
    return check_launch("forward");
}

flp_status fused_logp_backward(const void* logits, int64_t n, int64_t v, int64_t ld,
                               const int64_t* targets, int64_t ignore_index, const float* lse,
                               const float* lse_lo, const float* grad, void* dlogits,
                               int64_t ld_out, flp_stream_t stream) {
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v < 1) return fail(FLP_EINVAL, "v must be >= 1 (got %lld)", (long long)v);
    if (ld < v) return fail(FLP_EINVAL, "ld (%lld) must be >= v (%lld)", (long long)ld, (long long)v);
    if (ld_out < v)
        return fail(FLP_EINVAL, "ld_out (%lld) must be >= v (%lld)", (long long)ld_out, (long long)v);
    if (n == 0) return ok();
    int64_t in_bytes, out_bytes;
    if (!span_bytes(n, v, ld, 2, &in_bytes) || !span_bytes(n, v, ld_out, 2, &out_bytes))
        return fail(FLP_EINVAL, "logits/dlogits extent overflows int64");
    const void* ptrs[] = {logits, targets, lse, grad, dlogits, lse_lo ? lse_lo : lse};
    const char* names[] = {"logits", "targets", "lse", "grad", "dlogits", "lse_lo"};
    int dev;
    flp_status st = common_device(6, ptrs, names, &dev);
    if (st != FLP_OK) return st;

    const uintptr_t xb = reinterpret_cast<uintptr_t>(logits);
    const uintptr_t db = reinterpret_cast<uintptr_t>(dlogits);
    const bool in_place = (xb == db) && (ld == ld_out);
    if (!in_place && xb < db + (uintptr_t)out_bytes && db < xb + (uintptr_t)in_bytes)
        return fail(FLP_EINVAL, "dlogits overlaps logits without being exactly in place");

    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;

    const uint16_t* x = static_cast<const uint16_t*>(logits);
    uint16_t* dx = static_cast<uint16_t*>(dlogits);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t segs = ceil_div(v, flp::kBwdSegCols);
    int64_t items;
    if (__builtin_mul_overflow(n, segs, &items)) return fail(FLP_EINVAL, "n * segments overflows");
    const int grid = grid_for(items);
    const bool vin = aligned16(x) && ld % 8 == 0;
    const bool vout = aligned16(dx) && ld_out % 8 == 0;
#define FLP_BWD(VI, VO, IP)                                                                   \
    flp::k_logp_bwd<VI, VO, IP><<<grid, flp::kBwdThreads, 0, s>>>(x, n, v, ld, targets,      \
                                                                  ignore_index, lse, lse_lo, grad, dx, \
                                                                  ld_out, segs)
    if (in_place) {
        if (vin) FLP_BWD(true, true, true);
        else FLP_BWD(false, false, true);
    } else if (vin && vout) FLP_BWD(true, true, false);
    else if (vin) FLP_BWD(true, false, false);
    else if (vout) FLP_BWD(false, true, false);
    else FLP_BWD(false, false, false);
#undef FLP_BWD
    return check_launch("backward");
}

flp_status logp_shard_partials(const void* shard_logits, int64_t n, int64_t ld_shard,
                               int64_t vocab_start, int64_t real_width, int64_t v_total,
                               const int64_t* targets, float* part_max, float* part_sum,
                               float* sel, flp_stream_t stream) {
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v_total < 1) return fail(FLP_EINVAL, "v_total must be >= 1");
    if (real_width < 1) return fail(FLP_EINVAL, "real_width must be >= 1");
    if (vocab_start < 0 || vocab_start + real_width > v_total)
        return fail(FLP_EINVAL, "shard [%lld, %lld) is outside the vocabulary [0, %lld)",
                    (long long)vocab_start, (long long)(vocab_start + real_width),
                    (long long)v_total);
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
    if (!span_bytes(n, real_width, ld_shard, 2, &bytes))
        return fail(FLP_EINVAL, "shard extent overflows int64");
    const void* ptrs[] = {shard_logits, targets, part_max, part_sum, sel};
    const char* names[] = {"shard_logits", "targets", "part_max", "part_sum", "sel"};
    int dev;
    flp_status st = common_device(5, ptrs, names, &dev);
    if (st != FLP_OK) return st;
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;

    const int tile0 = (int)(vocab_start / W);
    const int ntile = (int)ceil_div(real_width, W);
    const uint16_t* xs = static_cast<const uint16_t*>(shard_logits);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int grid = grid_for(n);
    if (aligned16(xs) && ld_shard % 8 == 0)
        flp::k_logp_partials<true><<<grid, ntile * flp::kWarp, 0, s>>>(
            xs, n, ld_shard, real_width, W, tile0, vocab_start, targets, part_max, part_sum, sel);
    else
        flp::k_logp_partials<false><<<grid, ntile * flp::kWarp, 0, s>>>(
            xs, n, ld_shard, real_width, W, tile0, vocab_start, targets, part_max, part_sum, sel);
    return check_launch("shard partials");
}

flp_status logp_merge_partials(const float* part_max, const float* part_sum, const float* sel,
                               const int64_t* targets, int64_t ignore_index, int64_t n,
                               int64_t v_total, float* logp, float* lse, float* lse_lo,
                               flp_stream_t stream) {
    if (n < 0) return fail(FLP_EINVAL, "n must be >= 0 (got %lld)", (long long)n);
    if (v_total < 1) return fail(FLP_EINVAL, "v_total must be >= 1");
    if (n == 0) return ok();
    const void* ptrs[] = {part_max, part_sum, sel, targets, logp, lse, lse_lo ? lse_lo : lse};
    const char* names[] = {"part_max", "part_sum", "sel", "targets", "logp", "lse", "lse_lo"};
    int dev;
    flp_status st = common_device(7, ptrs, names, &dev);
    if (st != FLP_OK) return st;
    DeviceGuard guard;
    if ((st = guard.enter(dev)) != FLP_OK) return st;

    const int64_t W = tile_width(v_total);
    const int n_tiles = (int)ceil_div(v_total, W);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rows_per_block = 256 / 16;
    const int grid = grid_for(ceil_div(n, rows_per_block));
    flp::k_logp_merge<<<grid, 256, 0, s>>>(part_max, part_sum, sel, targets, ignore_index, n,
                                           v_total, n_tiles, logp, lse, lse_lo);
    return check_launch("merge");
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
