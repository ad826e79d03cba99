// vq_encode.cu -- C ABI entry points of the product-VQ encoder (see
// include/vq_encode.h for the contract of every function).
//
// Host side only: validate arguments, pick a kernel for the shape, launch it
// on the caller's stream.  The library allocates no memory.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "vq_encode.h"
#include "vq_host.h"
#include "vq_decode.cuh"
#include "vq_filter.cuh"
#include "vq_tc.cuh"
#include "vq_kernels.cuh"
#include "vq_status.cuh"

// Declared in vq_host.h.
int vqh_device_sms()
{
    constexpr int kMax = 64;
    // per device; concurrent first calls store the same value
    static std::atomic<int> cache[kMax] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMax) {
        (void)cudaGetLastError();
        return 0;
    }
    int sms = cache[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        cache[dev].store(sms, std::memory_order_relaxed);
    }
    return sms;
}

VQH_STATUS_READER(vqh_status_encode)

namespace {

// Tuning of the exact brute-force kernel (rows per thread, threads per block,
// argmin strategy, centroids per group).
constexpr int kThreads = 128;
constexpr int kRows = 8;
constexpr int kMode = vqk::kDeferred;
constexpr int kGroupCentroids = 8;
// Tuning of the filter-and-refine kernel.
constexpr int kFThreads = 128;
constexpr int kFRows = 8;
constexpr int kFGroup = 16;
// Tuning of the tensor-core screening kernel: vqk::TcConfig (vq_tc.cuh).
using vqk::TcConfig;

int device_sms() { return vqh_device_sms(); }

// Blocks per group and 128-row tiles per block.  A block works through its
// tiles `tps` at a time; its time is taken as its steps plus half a step of
// set-up (codebook staging), the launch's time as waves of `slots` resident
// blocks times that.  The best of 1..64 tiles per block and the one-wave
// shape is used.
void tc_shape(int64_t n_groups, int64_t n_per_group, int slots, int tps, int64_t *blocks_per_group,
              int32_t *tiles_per_block)
{
    const int64_t tiles = (n_per_group + 127) / 128;
    int64_t per_group = slots / n_groups;
    if (per_group < 1) per_group = 1;
    const int64_t one_wave = (tiles + per_group - 1) / per_group;
    int64_t best_t = 1;
    double best_cost = 1e300;
    auto consider = [&](int64_t t) {
        if (t < 1 || t > tiles) return;
        const int64_t blocks = n_groups * ((tiles + t - 1) / t);
        const int64_t waves = (blocks + slots - 1) / slots;
        const double cost = (double)waves * ((double)((t + tps - 1) / tps) + 0.5);
        if (cost < best_cost) {
            best_cost = cost;
            best_t = t;
        }
    };
    consider(one_wave);
    for (int64_t t = 1; t <= 64; ++t) consider(t);
    if (best_t > (1 << 30)) best_t = 1 << 30;
    *tiles_per_block = (int32_t)best_t;
    *blocks_per_group = (tiles + best_t - 1) / best_t;
}

// Codebooks smaller than this many centroids are brute-forced: screening pays
// off only with several centroid groups to rule out.
constexpr int kFilterMinCentroids = 4 * kFGroup;

constexpr int kMaxSubDim = 32;
constexpr int kMaxCentroids = 4096;
constexpr size_t kMaxFastSmem = 200 * 1024;
constexpr int kGeneralThreads = 128;

struct Args {
    const void *x;
    const void *cb;
    int64_t n_groups;
    int64_t n_per_group;
    int32_t n_centroids;
    int32_t sub_dim;
    vq_dtype dtype;
    void *out;
    cudaStream_t stream;
    int out_bytes = 4;  // index width: 4 (uint32) or 1 (uint8 codes)
    const float *smooth = nullptr;  // per-channel smooth factors [n_groups][head_dim]
    int32_t head_dim = 0;
};

size_t elem_size(vq_dtype d) { return d == VQ_F32 ? 4 : 2; }

vq_status validate(const Args &a, bool need_pointers)
{
    if (a.dtype != VQ_F16 && a.dtype != VQ_BF16 && a.dtype != VQ_F32) return VQ_ERR_INVALID_ARG;
    if (a.n_groups < 0 || a.n_per_group < 0) return VQ_ERR_INVALID_ARG;
    if (a.sub_dim < 1 || a.sub_dim > kMaxSubDim) return VQ_ERR_UNSUPPORTED;
    if (a.n_centroids < 1 || a.n_centroids > kMaxCentroids) return VQ_ERR_UNSUPPORTED;
    if (a.out_bytes == 1 && a.n_centroids > 256) return VQ_ERR_UNSUPPORTED;  // 8-bit codes
    if (a.n_groups != 0 && a.n_per_group > INT64_MAX / a.n_groups) return VQ_ERR_INVALID_ARG;
    const int64_t rows = a.n_groups * a.n_per_group;
    if (rows == 0) return VQ_OK;
    if (rows > INT64_MAX / (a.sub_dim * 4)) return VQ_ERR_INVALID_ARG;
    if (need_pointers) {
        if (!a.x || !a.cb || !a.out) return VQ_ERR_INVALID_ARG;
        const size_t es = elem_size(a.dtype);
        if ((uintptr_t)a.x % es || (uintptr_t)a.cb % es || (uintptr_t)a.out % a.out_bytes)
            return VQ_ERR_INVALID_ARG;
    }
    return VQ_OK;
}

enum KernelKind { kGeneral = 0, kBrute = 1, kFilter = 2, kTc = 3 };

struct Plan {
    KernelKind kind;
    size_t smem;
    int64_t tiles_per_group;  // blocks per group
    int64_t blocks;
    int threads;
    int32_t tc_tiles;         // 128-row tiles per block (tensor-core kernel)
};

template <int SUB>
size_t fast_smem(int32_t n_centroids)
{
    return vqk::CbLayout<SUB, kGroupCentroids>::bytes(n_centroids);
}

// A holds two tf32 pieces of each row when the rows are not 16-bit values
// (smoothed or fp32), B two pieces of -2c for fp32 codebooks.
template <int SUB, bool SMOOTH = false>
size_t tc_smem(int32_t n_centroids, vq_dtype dtype)
{
    if (dtype == VQ_F32) {
        using C = TcConfig<SUB, true>;
        return vqk::TcLayout<SUB, C::kCols, C::kGroup, 2, 2, C::kTps>::bytes(n_centroids);
    }
    using C = TcConfig<SUB, SMOOTH>;
    return vqk::TcLayout<SUB, C::kCols, C::kGroup, SMOOTH ? 2 : 1, 1, C::kTps>::bytes(n_centroids);
}

// Rows go to the tensor cores as two tf32 pieces when they are smoothed or fp32.
template <typename T, bool SMOOTH>
constexpr bool tc_split() { return SMOOTH || std::is_same<T, float>::value; }

template <typename T, int SUB, typename OutT = uint32_t, bool SMOOTH = false>
auto tc_kernel()
{
    using C = TcConfig<SUB, tc_split<T, SMOOTH>()>;
    return vqk::encode_tc<T, SUB, C::kCols, C::kGroup, C::kMinBlocks, OutT, SMOOTH, vqk::kWaitPolls, C::kTps>;
}

// Resident tensor-core CTAs on the device: the register budget of the launch
// bounds admits kMinBlocks per SM, the tensor memory 512 / kCols, and the
// shared memory of an SM (228 KiB, 1 KiB reserved per block) what `smem`
// allows.
// Tiles per step of the tensor-core kernel; `split` as in tc_split.
int tc_tps(int sub_dim, bool split)
{
    if (sub_dim == 4) return split ? TcConfig<4, true>::kTps : TcConfig<4, false>::kTps;
    return split ? TcConfig<8, true>::kTps : TcConfig<8, false>::kTps;
}

int tc_slots(int sub_dim, bool split, size_t smem)
{
    const int sms = device_sms();
    int per_sm = sub_dim == 4 ? (split ? TcConfig<4, true>::kMinBlocks : TcConfig<4, false>::kMinBlocks)
                              : (split ? TcConfig<8, true>::kMinBlocks : TcConfig<8, false>::kMinBlocks);
    const int by_smem = (int)((size_t)228 * 1024 / (smem + 1024));
    if (by_smem < per_sm) per_sm = by_smem;
    if (per_sm < 1) per_sm = 1;
    return (sms > 0 ? sms : 152) * per_sm;
}

template <int SUB>
size_t filter_smem(int32_t n_centroids)
{
    return vqk::FilterLayout<SUB, kFGroup>::bytes(n_centroids, kFThreads * kFRows);
}

Plan make_plan(const Args &a)
{
    Plan p{};
    const size_t es = elem_size(a.dtype);
    const size_t row_bytes = (size_t)a.sub_dim * es;
    const size_t align = row_bytes < 16 ? row_bytes : 16;
    const bool shape_ok = (a.sub_dim == 4 || a.sub_dim == 8) && ((uintptr_t)a.x % align == 0);
    p.kind = kGeneral;
    // tf32 holds fp16 and bf16 values exactly; fp32 rows and codebooks are
    // split into tf32 pieces, the dropped bits covered by the bound
    if (shape_ok && a.n_centroids >= kFilterMinCentroids && a.n_centroids <= 256) {
        p.kind = kTc;
        p.smem = a.sub_dim == 4 ? tc_smem<4>(a.n_centroids, a.dtype) : tc_smem<8>(a.n_centroids, a.dtype);
    }
    if (shape_ok && p.kind == kGeneral && a.n_centroids >= kFilterMinCentroids) {
        p.smem = a.sub_dim == 4 ? filter_smem<4>(a.n_centroids) : filter_smem<8>(a.n_centroids);
        if (p.smem <= kMaxFastSmem) p.kind = kFilter;
    }
    if (shape_ok && p.kind == kGeneral) {
        p.smem = a.sub_dim == 4 ? fast_smem<4>(a.n_centroids) : fast_smem<8>(a.n_centroids);
        if (p.smem <= kMaxFastSmem) p.kind = kBrute;
    }
    if (p.kind == kTc) {
        const bool split = a.dtype == VQ_F32;
        tc_shape(a.n_groups, a.n_per_group, tc_slots(a.sub_dim, split, p.smem), tc_tps(a.sub_dim, split),
                 &p.tiles_per_group, &p.tc_tiles);
        p.blocks = a.n_groups * p.tiles_per_group;
        p.threads = 128 * tc_tps(a.sub_dim, split);
    } else if (p.kind != kGeneral) {
        const int64_t tile = p.kind == kFilter ? (int64_t)kFThreads * kFRows : (int64_t)kThreads * kRows;
        p.tiles_per_group = (a.n_per_group + tile - 1) / tile;
        p.blocks = a.n_groups * p.tiles_per_group;
        p.threads = p.kind == kFilter ? kFThreads : kThreads;
    } else {
        p.smem = 0;
        p.tiles_per_group = 0;
        p.blocks = (a.n_groups * a.n_per_group + kGeneralThreads - 1) / kGeneralThreads;
        p.threads = kGeneralThreads;
    }
    return p;
}

template <typename T, int SUB, typename OutT, bool SMOOTH = false>
vq_status launch_tc(const Args &a, const Plan &p)
{
    auto kernel = tc_kernel<T, SUB, OutT, SMOOTH>();
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) !=
        cudaSuccess)
        return VQ_ERR_CUDA;
    kernel<<<(unsigned)p.blocks, 128 * TcConfig<SUB, tc_split<T, SMOOTH>()>::kTps, p.smem, a.stream>>>(
        static_cast<const T *>(a.x), static_cast<const T *>(a.cb), a.n_per_group, a.n_centroids,
        p.tiles_per_group, p.tc_tiles, 1.0f, static_cast<OutT *>(a.out), a.smooth,
        SMOOTH ? (int32_t)(a.head_dim / a.sub_dim) : 1);
    return vqh_launched(a.stream, vqh_status_encode);
}

template <typename T, int SUB, typename OutT, bool SMOOTH = false>
vq_status launch_filter(const Args &a, const Plan &p)
{
    auto kernel = vqk::encode_filter<T, SUB, kFRows, kFThreads, kFGroup, OutT, SMOOTH>;
    if (p.smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)p.smem) != cudaSuccess)
            return VQ_ERR_CUDA;
    }
    kernel<<<(unsigned)p.blocks, p.threads, p.smem, a.stream>>>(
        static_cast<const T *>(a.x), static_cast<const T *>(a.cb), a.n_per_group, a.n_centroids,
        p.tiles_per_group, 1.0f, static_cast<OutT *>(a.out), a.smooth,
        SMOOTH ? a.head_dim / SUB : 0);
    return vqh_launched(a.stream, vqh_status_encode);
}

template <typename T, int SUB, typename OutT>
vq_status launch_fast(const Args &a, const Plan &p)
{
    auto kernel = vqk::encode_fast<T, SUB, kRows, kThreads, kMode, kGroupCentroids, OutT>;
    if (p.smem > 48 * 1024) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)p.smem) != cudaSuccess)
            return VQ_ERR_CUDA;
    }
    kernel<<<(unsigned)p.blocks, p.threads, p.smem, a.stream>>>(
        static_cast<const T *>(a.x), static_cast<const T *>(a.cb), a.n_per_group, a.n_centroids,
        p.tiles_per_group, 1.0f, static_cast<OutT *>(a.out));
    return vqh_launched(a.stream, vqh_status_encode);
}

template <typename T, typename OutT>
vq_status launch_general(const Args &a, const Plan &p)
{
    vqk::encode_general<T, OutT><<<(unsigned)p.blocks, p.threads, 0, a.stream>>>(
        static_cast<const T *>(a.x), static_cast<const T *>(a.cb), a.n_groups, a.n_per_group,
        a.n_centroids, a.sub_dim, 1.0f, static_cast<OutT *>(a.out));
    return vqh_launched(a.stream, vqh_status_encode);
}

template <typename T, typename OutT>
vq_status launch_typed(const Args &a, const Plan &p)
{
    switch (p.kind) {
    case kTc:
        return a.sub_dim == 4 ? launch_tc<T, 4, OutT>(a, p) : launch_tc<T, 8, OutT>(a, p);
    case kFilter:
        return a.sub_dim == 4 ? launch_filter<T, 4, OutT>(a, p) : launch_filter<T, 8, OutT>(a, p);
    case kBrute:
        return a.sub_dim == 4 ? launch_fast<T, 4, OutT>(a, p) : launch_fast<T, 8, OutT>(a, p);
    case kGeneral: return launch_general<T, OutT>(a, p);
    }
    return VQ_ERR_INTERNAL;
}

template <typename OutT>
vq_status launch_dtype(const Args &a, const Plan &p)
{
    switch (a.dtype) {
    case VQ_F16: return launch_typed<__half, OutT>(a, p);
    case VQ_BF16: return launch_typed<__nv_bfloat16, OutT>(a, p);
    case VQ_F32: return launch_typed<float, OutT>(a, p);
    }
    return VQ_ERR_INTERNAL;
}

vq_status run(const Args &a)
{
    vq_status s = validate(a, true);
    if (s != VQ_OK) return s;
    if (a.n_groups * a.n_per_group == 0) return VQ_OK;
    const Plan p = make_plan(a);
    if (p.blocks > 0x7fffffffLL) return VQ_ERR_UNSUPPORTED;
    return a.out_bytes == 1 ? launch_dtype<uint8_t>(a, p) : launch_dtype<uint32_t>(a, p);
}

template <typename OutT, int SUB>
vq_status launch_smooth_typed(const Args &a, const Plan &p)
{
    if (p.kind == kTc) {
        switch (a.dtype) {
        case VQ_F16: return launch_tc<__half, SUB, OutT, true>(a, p);
        case VQ_BF16: return launch_tc<__nv_bfloat16, SUB, OutT, true>(a, p);
        case VQ_F32: return launch_tc<float, SUB, OutT, true>(a, p);
        default: return VQ_ERR_INTERNAL;
        }
    }
    switch (a.dtype) {
    case VQ_F16: return launch_filter<__half, SUB, OutT, true>(a, p);
    case VQ_BF16: return launch_filter<__nv_bfloat16, SUB, OutT, true>(a, p);
    case VQ_F32: return launch_filter<float, SUB, OutT, true>(a, p);
    }
    return VQ_ERR_INTERNAL;
}

// Encode with per-channel smoothing.  Codebooks of 64..256 centroids take the
// tensor-core kernel with the divided rows split into two tf32 pieces (and
// fp32 codebooks too; the bound covers the dropped low bits); others the
// filter kernel, whose bound holds for any fp32 row.
vq_status run_smooth(const Args &a)
{
    if (a.head_dim < a.sub_dim || a.sub_dim < 1 || a.head_dim % a.sub_dim) return VQ_ERR_INVALID_ARG;
    if (a.n_per_group >= 0 && a.n_per_group % (a.head_dim / a.sub_dim)) return VQ_ERR_INVALID_ARG;
    vq_status s = validate(a, true);
    if (s != VQ_OK) return s;
    if (a.n_groups * a.n_per_group == 0) return VQ_OK;
    if (a.sub_dim != 4 && a.sub_dim != 8) return VQ_ERR_UNSUPPORTED;
    if (!a.smooth || (uintptr_t)a.smooth % sizeof(float)) return VQ_ERR_INVALID_ARG;
    const size_t row_bytes = (size_t)a.sub_dim * elem_size(a.dtype);
    if ((uintptr_t)a.x % (row_bytes < 16 ? row_bytes : 16)) return VQ_ERR_UNSUPPORTED;
    Plan p{};
    if (a.n_centroids >= kFilterMinCentroids && a.n_centroids <= 256) {
        p.kind = kTc;
        p.smem = a.sub_dim == 4 ? tc_smem<4, true>(a.n_centroids, a.dtype) : tc_smem<8, true>(a.n_centroids, a.dtype);
        tc_shape(a.n_groups, a.n_per_group, tc_slots(a.sub_dim, true, p.smem), tc_tps(a.sub_dim, true),
                 &p.tiles_per_group, &p.tc_tiles);
        p.blocks = a.n_groups * p.tiles_per_group;
        p.threads = 128 * tc_tps(a.sub_dim, true);
    } else {
        p.kind = kFilter;
        p.smem = a.sub_dim == 4 ? filter_smem<4>(a.n_centroids) : filter_smem<8>(a.n_centroids);
        if (p.smem > kMaxFastSmem) return VQ_ERR_UNSUPPORTED;
        const int64_t tile = (int64_t)kFThreads * kFRows;
        p.tiles_per_group = (a.n_per_group + tile - 1) / tile;
        p.blocks = a.n_groups * p.tiles_per_group;
        p.threads = kFThreads;
    }
    if (p.blocks > 0x7fffffffLL) return VQ_ERR_UNSUPPORTED;
    if (a.out_bytes == 1)
        return a.sub_dim == 4 ? launch_smooth_typed<uint8_t, 4>(a, p) : launch_smooth_typed<uint8_t, 8>(a, p);
    return a.sub_dim == 4 ? launch_smooth_typed<uint32_t, 4>(a, p) : launch_smooth_typed<uint32_t, 8>(a, p);
}

const char *dtype_name(vq_dtype d)
{
    switch (d) {
    case VQ_F16: return "f16";
    case VQ_BF16: return "bf16";
    case VQ_F32: return "f32";
    }
    return "?";
}

// Per-device copy streams and events of the host entry point's copy path,
// created on the first such call on a device and kept until exit.  The mutex
// serialises host calls on one device, which share them.
constexpr int kMaxDevices = 64;
constexpr int kHostChunks = 4;
constexpr int kHostEvents = 8;
// A chunk must fill the GPU several times over, or its encode runs below
// full occupancy and the overlap gains nothing.
constexpr int64_t kHostChunkMinRows = int64_t(1) << 22;

struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t loaded[kHostEvents] = {}, encoded[kHostEvents] = {}, copied[kHostEvents] = {};

    vq_status init()
    {
        const unsigned ev_flags = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&start, ev_flags) == cudaSuccess;
        for (int i = 0; ok && i < kHostEvents; ++i)
            ok = cudaEventCreateWithFlags(&loaded[i], ev_flags) == cudaSuccess &&
                 cudaEventCreateWithFlags(&encoded[i], ev_flags) == cudaSuccess &&
                 cudaEventCreateWithFlags(&copied[i], ev_flags) == cudaSuccess;
        ready = ok;
        return ok ? VQ_OK : VQ_ERR_CUDA;
    }
};

HostPipe host_pipes[kMaxDevices];

// The device-side address of a host pointer, if the GPU can access it
// (page-locked host memory on a unified-address system).
bool device_view(const void *p, void **dptr)
{
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();  // not a CUDA-known pointer: clear the non-sticky error
        return false;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return false;
    *dptr = at.devicePointer;
    return true;
}

}  // namespace

extern "C" {

vq_status vq_encode(const void *x, const void *codebook, int64_t n, int32_t n_centroids,
                    int32_t sub_dim, vq_dtype dtype, uint32_t *out_idx, vq_stream_t stream)
{
    if (n < 0) return VQ_ERR_INVALID_ARG;
    return run(Args{x, codebook, 1, n, n_centroids, sub_dim, dtype, out_idx,
                    reinterpret_cast<cudaStream_t>(stream)});
}

vq_status vq_encode_grouped(const void *x, const void *codebooks, int64_t n_groups,
                            int64_t n_per_group, int32_t n_centroids, int32_t sub_dim,
                            vq_dtype dtype, uint32_t *out_idx, vq_stream_t stream)
{
    return run(Args{x, codebooks, n_groups, n_per_group, n_centroids, sub_dim, dtype, out_idx,
                    reinterpret_cast<cudaStream_t>(stream)});
}

vq_status vq_encode_grouped_host(const void *x_host, const void *codebooks_host,
                                 int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                                 int32_t sub_dim, vq_dtype dtype, uint32_t *out_host,
                                 void *x_dev, void *codebooks_dev, uint32_t *out_dev,
                                 vq_stream_t stream)
{
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Args a{x_dev, codebooks_dev, n_groups, n_per_group, n_centroids, sub_dim, dtype, out_dev, st};
    vq_status s = validate(a, true);
    if (s != VQ_OK) return s;
    const int64_t rows = n_groups * n_per_group;
    if (rows == 0) return VQ_OK;
    if (!x_host || !codebooks_host || !out_host) return VQ_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    const size_t cb_bytes = (size_t)n_groups * n_centroids * sub_dim * es;

    // Pinned (page-locked, mapped) host buffers are addressable by the GPU: on
    // GB300 the kernel then reads x and writes the indices across the
    // coherent CPU-GPU link while it computes, with no staging copies.  Only
    // the codebooks (a few KiB per group) are copied to the device.
    void *x_view = nullptr, *out_view = nullptr;
    if (device_view(x_host, &x_view) && device_view(out_host, &out_view)) {
        if (cudaMemcpyAsync(codebooks_dev, codebooks_host, cb_bytes, cudaMemcpyHostToDevice, st) !=
            cudaSuccess)
            return VQ_ERR_CUDA;
        Args z{x_view, codebooks_dev, n_groups, n_per_group, n_centroids, sub_dim, dtype,
               out_view, st};
        s = run(z);
        if (s != VQ_OK) return s;
        return cudaStreamSynchronize(st) == cudaSuccess ? VQ_OK : VQ_ERR_CUDA;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VQ_ERR_CUDA;
    HostPipe &hp = host_pipes[dev];
    std::lock_guard<std::mutex> guard(hp.mu);
    if (!hp.ready && (s = hp.init()) != VQ_OK) return s;

    const size_t row_bytes = (size_t)sub_dim * es;
    const size_t cb_group_bytes = (size_t)n_centroids * sub_dim * es;
    const char *xh = static_cast<const char *>(x_host);
    char *xd = static_cast<char *>(x_dev);
    const char *cbd = static_cast<const char *>(codebooks_dev);

    // Chunks: whole groups when there are many, else equal row ranges of each
    // group; never smaller than kHostChunkMinRows rows.
    const int64_t want = std::max<int64_t>(1, std::min<int64_t>(kHostChunks, rows / kHostChunkMinRows));
    const int64_t groups_per_chunk = n_groups >= want ? (n_groups + want - 1) / want : 1;
    const int64_t splits = n_groups >= want ? 1 : (want + n_groups - 1) / n_groups;
    const int64_t rows_per_split = (n_per_group + splits - 1) / splits;

    // The copy streams must not overwrite device buffers still in use by work
    // already queued on the caller's stream.
    bool ok = cudaEventRecord(hp.start, st) == cudaSuccess &&
              cudaStreamWaitEvent(hp.h2d, hp.start, 0) == cudaSuccess &&
              cudaMemcpyAsync(codebooks_dev, codebooks_host, cb_bytes, cudaMemcpyHostToDevice,
                              hp.h2d) == cudaSuccess;
    int ci = 0;
    for (int64_t g0 = 0; ok && g0 < n_groups; g0 += groups_per_chunk) {
        const int64_t ng = std::min(groups_per_chunk, n_groups - g0);
        for (int64_t r0 = 0; ok && r0 < n_per_group; r0 += rows_per_split) {
            const int64_t nr = std::min(rows_per_split, n_per_group - r0);
            const int slot = ci % kHostEvents;
            // rows [g0*M + r0, ...): with splits == 1 the chunk is ng whole groups
            const int64_t first = g0 * n_per_group + r0;
            const int64_t count = splits == 1 ? ng * n_per_group : nr;
            if (ci >= kHostEvents)  // slot reuse: its previous copy back must be done
                ok = cudaEventSynchronize(hp.copied[slot]) == cudaSuccess;
            ok = ok &&
                 cudaMemcpyAsync(xd + first * row_bytes, xh + first * row_bytes,
                                 (size_t)count * row_bytes, cudaMemcpyHostToDevice,
                                 hp.h2d) == cudaSuccess &&
                 cudaEventRecord(hp.loaded[slot], hp.h2d) == cudaSuccess &&
                 cudaStreamWaitEvent(st, hp.loaded[slot], 0) == cudaSuccess;
            if (!ok) break;
            Args c{xd + first * row_bytes, cbd + g0 * cb_group_bytes, splits == 1 ? ng : 1,
                   splits == 1 ? n_per_group : nr, n_centroids, sub_dim, dtype, out_dev + first, st};
            s = run(c);
            if (s != VQ_OK) return s;
            ok = cudaEventRecord(hp.encoded[slot], st) == cudaSuccess &&
                 cudaStreamWaitEvent(hp.d2h, hp.encoded[slot], 0) == cudaSuccess &&
                 cudaMemcpyAsync(out_host + first, out_dev + first, (size_t)count * 4,
                                 cudaMemcpyDeviceToHost, hp.d2h) == cudaSuccess &&
                 cudaEventRecord(hp.copied[slot], hp.d2h) == cudaSuccess;
            ++ci;
            if (splits == 1) break;
        }
    }
    // The caller's stream ends after the last copy back; return once it is done.
    ok = ok && cudaEventRecord(hp.start, hp.d2h) == cudaSuccess &&
         cudaStreamWaitEvent(st, hp.start, 0) == cudaSuccess &&
         cudaStreamSynchronize(hp.d2h) == cudaSuccess;
    return ok ? VQ_OK : VQ_ERR_CUDA;
}

vq_status vq_encode_grouped_u8(const void *x, const void *codebooks, int64_t n_groups,
                               int64_t n_per_group, int32_t n_centroids, int32_t sub_dim,
                               vq_dtype dtype, uint8_t *out_idx, vq_stream_t stream)
{
    Args a{x, codebooks, n_groups, n_per_group, n_centroids, sub_dim, dtype, out_idx,
           reinterpret_cast<cudaStream_t>(stream)};
    a.out_bytes = 1;
    return run(a);
}

vq_status vq_encode_grouped_smooth(const void *x, const float *smooth, const void *codebooks,
                                   int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                                   int32_t sub_dim, int32_t head_dim, vq_dtype dtype, void *out_idx,
                                   int32_t index_bytes, vq_stream_t stream)
{
    if (index_bytes != 1 && index_bytes != 4) return VQ_ERR_INVALID_ARG;
    Args a{x, codebooks, n_groups, n_per_group, n_centroids, sub_dim, dtype, out_idx,
           reinterpret_cast<cudaStream_t>(stream)};
    a.out_bytes = index_bytes;
    a.smooth = smooth;
    a.head_dim = head_dim;
    return run_smooth(a);
}

vq_status vq_dequantize_grouped(const void *idx, int32_t index_bytes, const void *codebooks,
                                int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                                int32_t sub_dim, vq_dtype dtype, void *out, vq_stream_t stream)
{
    if (dtype != VQ_F16 && dtype != VQ_BF16 && dtype != VQ_F32) return VQ_ERR_INVALID_ARG;
    if (index_bytes != 1 && index_bytes != 4) return VQ_ERR_INVALID_ARG;
    if (n_groups < 0 || n_per_group < 0) return VQ_ERR_INVALID_ARG;
    if (sub_dim < 1 || sub_dim > kMaxSubDim) return VQ_ERR_UNSUPPORTED;
    if (n_centroids < 1 || n_centroids > kMaxCentroids) return VQ_ERR_UNSUPPORTED;
    if (n_groups != 0 && n_per_group > INT64_MAX / n_groups) return VQ_ERR_INVALID_ARG;
    const int64_t rows = n_groups * n_per_group;
    if (rows == 0) return VQ_OK;
    if (rows > INT64_MAX / (sub_dim * 4)) return VQ_ERR_INVALID_ARG;
    if (!idx || !codebooks || !out) return VQ_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if ((uintptr_t)idx % index_bytes || (uintptr_t)codebooks % es || (uintptr_t)out % es)
        return VQ_ERR_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t row_bytes = (size_t)sub_dim * es;
    const size_t align = row_bytes < 16 ? row_bytes : 16;
    const bool fast = (row_bytes == 8 || row_bytes == 16 || row_bytes == 32) &&
                      (uintptr_t)codebooks % align == 0 && (uintptr_t)out % align == 0;
    if (fast) {
        constexpr int kT = 256, kR = 8;
        const int64_t per_group = (n_per_group + kT * kR - 1) / (kT * kR);
        const int64_t blocks = n_groups * per_group;
        if (blocks > 0x7fffffffLL) return VQ_ERR_UNSUPPORTED;
        const auto *cb = static_cast<const unsigned char *>(codebooks);
        auto *o = static_cast<unsigned char *>(out);
        const unsigned nb = (unsigned)blocks;
#define VQ_DECODE(IDXT, BYTES)                                                                     \
    vqk::decode_rows<IDXT, BYTES, kT, kR><<<nb, kT, 0, st>>>(static_cast<const IDXT *>(idx), cb,     \
                                                            n_per_group, n_centroids, per_group, o)
        if (index_bytes == 4) {
            if (row_bytes == 8) VQ_DECODE(uint32_t, 8);
            else if (row_bytes == 16) VQ_DECODE(uint32_t, 16);
            else VQ_DECODE(uint32_t, 32);
        } else {
            if (row_bytes == 8) VQ_DECODE(uint8_t, 8);
            else if (row_bytes == 16) VQ_DECODE(uint8_t, 16);
            else VQ_DECODE(uint8_t, 32);
        }
#undef VQ_DECODE
    } else {
        constexpr int kT = 256;
        const int64_t total = rows * sub_dim;
        const int64_t blocks = (total + kT - 1) / kT;
        if (blocks > 0x7fffffffLL) return VQ_ERR_UNSUPPORTED;
        const unsigned nb = (unsigned)blocks;
        if (es == 2) {
            if (index_bytes == 4)
                vqk::decode_elems<uint32_t, uint16_t><<<nb, kT, 0, st>>>(
                    static_cast<const uint32_t *>(idx), static_cast<const uint16_t *>(codebooks),
                    n_groups, n_per_group, n_centroids, sub_dim, static_cast<uint16_t *>(out));
            else
                vqk::decode_elems<uint8_t, uint16_t><<<nb, kT, 0, st>>>(
                    static_cast<const uint8_t *>(idx), static_cast<const uint16_t *>(codebooks),
                    n_groups, n_per_group, n_centroids, sub_dim, static_cast<uint16_t *>(out));
        } else {
            if (index_bytes == 4)
                vqk::decode_elems<uint32_t, uint32_t><<<nb, kT, 0, st>>>(
                    static_cast<const uint32_t *>(idx), static_cast<const uint32_t *>(codebooks),
                    n_groups, n_per_group, n_centroids, sub_dim, static_cast<uint32_t *>(out));
            else
                vqk::decode_elems<uint8_t, uint32_t><<<nb, kT, 0, st>>>(
                    static_cast<const uint8_t *>(idx), static_cast<const uint32_t *>(codebooks),
                    n_groups, n_per_group, n_centroids, sub_dim, static_cast<uint32_t *>(out));
        }
    }
    return vqh_launched(st, vqh_status_encode);
}

vq_status vq_partition(int64_t n_groups, int64_t n_per_group, int32_t world, int32_t rank,
                       vq_slice *slices, int32_t *n_slices)
{
    if (!slices || !n_slices || world < 1 || rank < 0 || rank >= world || n_groups < 0 ||
        n_per_group < 0)
        return VQ_ERR_INVALID_ARG;
    if (n_groups != 0 && n_per_group > INT64_MAX / n_groups) return VQ_ERR_INVALID_ARG;
    *n_slices = 0;
    const int64_t total = n_groups * n_per_group;
    // floor(r T / world) without overflow: r (T / world) + floor(r (T % world) / world)
    const int64_t q = total / world, rem = total % world;
    auto start = [&](int64_t r) { return r * q + (r * rem) / world; };
    const int64_t s = start(rank), e = start((int64_t)rank + 1);
    if (s >= e) return VQ_OK;
    const int64_t m = n_per_group;
    const int64_t gs = s / m, rs = s % m, ge = e / m, re = e % m;
    int32_t k = 0;
    if (gs == ge) {  // inside one group
        slices[k++] = vq_slice{gs, 1, rs, re - rs};
    } else {
        int64_t full = gs;
        if (rs > 0) {  // the end of the first group
            slices[k++] = vq_slice{gs, 1, rs, m - rs};
            full = gs + 1;
        }
        if (ge > full) slices[k++] = vq_slice{full, ge - full, 0, m};  // whole groups
        if (re > 0) slices[k++] = vq_slice{ge, 1, 0, re};  // the start of the last
    }
    *n_slices = k;
    return VQ_OK;
}

const char *vq_status_string(vq_status status)
{
    switch (status) {
    case VQ_OK: return "VQ_OK: success";
    case VQ_ERR_INVALID_ARG: return "VQ_ERR_INVALID_ARG: invalid argument";
    case VQ_ERR_UNSUPPORTED: return "VQ_ERR_UNSUPPORTED: sub_dim or n_centroids not supported";
    case VQ_ERR_CUDA: return "VQ_ERR_CUDA: a CUDA call or kernel launch failed";
    case VQ_ERR_INTERNAL: return "VQ_ERR_INTERNAL: internal error";
    }
    return "unknown vq_status";
}

vq_status vq_describe_launch(int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                             int32_t sub_dim, vq_dtype dtype, const void *x, char *buf,
                             int32_t buflen)
{
    Args a{x, nullptr, n_groups, n_per_group, n_centroids, sub_dim, dtype, nullptr, nullptr};
    vq_status s = validate(a, false);
    if (s != VQ_OK) return s;
    if (!buf || buflen <= 0) return VQ_ERR_INVALID_ARG;
    // without a usable GPU the tensor-core kernel's shape assumes 152 SMs
    const Plan p = make_plan(a);
    if (p.kind == kTc)
        snprintf(buf, (size_t)buflen,
                 "kernel=encode_tc dtype=%s sub_dim=%d tmem_cols=%d tiles_per_block=%d "
                 "tiles_per_step=%d centroid_group=%d grid=%lld smem=%zu",
                 dtype_name(dtype), sub_dim, sub_dim == 4 ? TcConfig<4>::kCols : TcConfig<8>::kCols,
                 (int)p.tc_tiles, tc_tps(sub_dim, dtype == VQ_F32), sub_dim == 4 ? TcConfig<4>::kGroup : TcConfig<8>::kGroup,
                 (long long)p.blocks, p.smem);
    else if (p.kind == kFilter)
        snprintf(buf, (size_t)buflen,
                 "kernel=encode_filter dtype=%s sub_dim=%d rows_per_thread=%d threads=%d "
                 "centroid_group=%d grid=%lld smem=%zu",
                 dtype_name(dtype), sub_dim, kFRows, kFThreads, kFGroup, (long long)p.blocks,
                 p.smem);
    else if (p.kind == kBrute)
        snprintf(buf, (size_t)buflen,
                 "kernel=encode_fast dtype=%s sub_dim=%d rows_per_thread=%d threads=%d "
                 "argmin=%s centroid_group=%d grid=%lld smem=%zu",
                 dtype_name(dtype), sub_dim, kRows, kThreads,
                 kMode == vqk::kDeferred ? "deferred" : "direct", kGroupCentroids,
                 (long long)p.blocks, p.smem);
    else
        snprintf(buf, (size_t)buflen, "kernel=encode_general dtype=%s sub_dim=%d threads=%d grid=%lld",
                 dtype_name(dtype), sub_dim, p.threads, (long long)p.blocks);
    return VQ_OK;
}

int32_t vq_abi_version(void) { return VQ_ENCODE_ABI_VERSION; }

vq_status vq_kernel_status(uint32_t *bits, int32_t clear)
{
    if (!bits) return VQ_ERR_INVALID_ARG;
    *bits = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return VQ_ERR_CUDA;
    const bool c = clear != 0;
    if (vqh_status_encode(bits, c) != cudaSuccess || vqh_status_attn(bits, c) != cudaSuccess ||
        vqh_status_scalar(bits, c) != cudaSuccess)
        return VQ_ERR_CUDA;
    return VQ_OK;
}

}  // extern "C"
