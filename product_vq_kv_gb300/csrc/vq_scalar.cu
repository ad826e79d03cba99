// vq_scalar.cu -- C ABI entry points of the sibling encoders: scalar
// (sub_dim = 1) quantize and dequantize, and the randomised Hadamard rotation
// with its fused quantize (see include/vq_encode.h for each contract).
//
// Host side only: validate, pick the kernel of vq_scalar.cuh, launch on the
// caller's stream.  The library allocates nothing.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "vq_encode.h"
#include "vq_host.h"
#include "vq_status.cuh"
#include "vq_scalar.cuh"

VQH_STATUS_READER(vqh_status_scalar)

namespace {

constexpr int kThreads = 256;
constexpr size_t kTableBytes = 65536;
constexpr int kLookupThreads = 1024;

bool dtype_ok(vq_dtype d) { return d == VQ_F16 || d == VQ_BF16 || d == VQ_F32; }
size_t elem_size(vq_dtype d) { return d == VQ_F32 ? 4 : 2; }

int64_t stream_blocks(int64_t work_items, int per_sm)
{
    const int sms = vqh_device_sms() > 0 ? vqh_device_sms() : 152;
    int64_t b = (work_items + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sms * per_sm;
    if (b > cap) b = cap;
    return b < 1 ? 1 : b;
}

// Status of the launches just made on `st` (vq_host.h).
vq_status launched(cudaStream_t st) { return vqh_launched(st, vqh_status_scalar); }

template <typename T, int NC>
vq_status launch_scan_nc(const void *x, int64_t n, const float *c, int32_t n_c, uint8_t *out,
                         cudaStream_t st)
{
    const size_t smem = NC == 0 ? vqs::hadamard_smem(n_c) : 0;
    const bool vec = (uintptr_t)x % 16 == 0 && (uintptr_t)out % 8 == 0;
    vqs::scalar_scan<T, NC><<<(unsigned)stream_blocks((n + 7) / 8, 8), kThreads, smem, st>>>(
        static_cast<const T *>(x), n, c, n_c, vec, out);
    return launched(st);
}

template <typename T>
vq_status launch_scan(const void *x, int64_t n, const float *c, int32_t n_c, uint8_t *out,
                      cudaStream_t st)
{
    switch (n_c) {
    case 2: return launch_scan_nc<T, 2>(x, n, c, n_c, out, st);
    case 4: return launch_scan_nc<T, 4>(x, n, c, n_c, out, st);
    case 8: return launch_scan_nc<T, 8>(x, n, c, n_c, out, st);
    case 16: return launch_scan_nc<T, 16>(x, n, c, n_c, out, st);
    }
    return launch_scan_nc<T, 0>(x, n, c, n_c, out, st);
}

template <typename T, int E, bool QUANT, int NC>
vq_status launch_hadamard_nc(const void *x, const float *diag, int64_t n_rows, int lpr,
                             float scale, const float *c, int32_t n_c, float *y, uint8_t *idx,
                             cudaStream_t st)
{
    const int64_t rows_per_block = (int64_t)(kThreads / 32) * (32 / lpr);
    int64_t blocks = (n_rows + rows_per_block - 1) / rows_per_block;
    const int sms = vqh_device_sms() > 0 ? vqh_device_sms() : 152;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    const size_t smem = QUANT && NC == 0 ? vqs::hadamard_smem(n_c) : 0;
    vqs::hadamard_rows<T, E, QUANT, NC><<<(unsigned)blocks, kThreads, smem, st>>>(
        static_cast<const T *>(x), diag, n_rows, lpr, scale, c, n_c, y, idx);
    return launched(st);
}

// Codebooks of 2, 4, 8 or 16 entries (the pages' 1- to 4-bit Lloyd-Max
// codebooks) are scanned from registers; others through the sorted view.
template <typename T, int E, bool QUANT>
vq_status launch_hadamard_e(const void *x, const float *diag, int64_t n_rows, int lpr, float scale,
                            const float *c, int32_t n_c, float *y, uint8_t *idx, cudaStream_t st)
{
    if constexpr (QUANT) {
        switch (n_c) {
        case 2: return launch_hadamard_nc<T, E, true, 2>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
        case 4: return launch_hadamard_nc<T, E, true, 4>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
        case 8: return launch_hadamard_nc<T, E, true, 8>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
        case 16: return launch_hadamard_nc<T, E, true, 16>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
        }
    }
    return launch_hadamard_nc<T, E, QUANT, 0>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
}

// Lanes per row: up to 32 with at least eight elements each (fewer shuffle
// stages, each stage's set-up spread over more elements) when x and the codes
// are aligned for runs of that length; otherwise the layout the contract's
// alignment guarantees: one element per lane up to dim 32, then dim / 32.
template <typename T, bool QUANT>
vq_status launch_hadamard_t(const void *x, const float *diag, int64_t n_rows, int32_t dim,
                            float scale, const float *c, int32_t n_c, float *y, uint8_t *idx,
                            cudaStream_t st)
{
    int lpr = dim < 32 ? dim : 32;
    const int lpr_w = dim >= 8 ? (dim / 8 < 32 ? dim / 8 : 32) : 1;
    const size_t run_w = (size_t)(dim / lpr_w) * sizeof(T);
    if ((uintptr_t)x % (run_w < 16 ? run_w : 16) == 0 &&
        (!QUANT || (dim / lpr_w) % 4 != 0 || (uintptr_t)idx % 4 == 0))
        lpr = lpr_w;
    switch (dim / lpr) {
    case 1: return launch_hadamard_e<T, 1, QUANT>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
    case 2: return launch_hadamard_e<T, 2, QUANT>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
    case 4: return launch_hadamard_e<T, 4, QUANT>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
    case 8: return launch_hadamard_e<T, 8, QUANT>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
    case 16: return launch_hadamard_e<T, 16, QUANT>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
    case 32: return launch_hadamard_e<T, 32, QUANT>(x, diag, n_rows, lpr, scale, c, n_c, y, idx, st);
    }
    return VQ_ERR_INTERNAL;
}

template <bool QUANT>
vq_status hadamard(const void *x, vq_dtype dtype, const float *diag, int64_t n_rows, int32_t dim,
                   const float *c, int32_t n_c, float *y, uint8_t *idx, vq_stream_t stream)
{
    if (!dtype_ok(dtype) || n_rows < 0) return VQ_ERR_INVALID_ARG;
    if (dim < 1 || (dim & (dim - 1))) return VQ_ERR_INVALID_ARG;
    if (dim > 1024) return VQ_ERR_UNSUPPORTED;
    if (QUANT && (n_c < 1 || n_c > 256)) return VQ_ERR_UNSUPPORTED;
    if (n_rows == 0) return VQ_OK;
    if (!x || !diag || (QUANT ? (!c || !idx) : !y)) return VQ_ERR_INVALID_ARG;
    if ((uintptr_t)x % elem_size(dtype) || (uintptr_t)diag % 4 || (QUANT && (uintptr_t)c % 4) ||
        (!QUANT && (uintptr_t)y % 4) || (QUANT && dim >= 128 && (uintptr_t)idx % 4))
        return VQ_ERR_INVALID_ARG;
    if (n_rows > INT64_MAX / dim) return VQ_ERR_INVALID_ARG;
    {  // the rotation kernel reads each lane's run of dim/32 elements as vectors
        const size_t run = (size_t)(dim >= 32 ? dim / 32 : 1) * elem_size(dtype);
        if ((uintptr_t)x % (run < 16 ? run : 16)) return VQ_ERR_INVALID_ARG;
    }
    // fp32 value of 1/sqrt(dim), correctly rounded (2^(-k/2) for dim = 2^k)
    const float scale = (float)(1.0 / std::sqrt((double)dim));
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (dtype) {
    case VQ_F16: return launch_hadamard_t<__half, QUANT>(x, diag, n_rows, dim, scale, c, n_c, y, idx, st);
    case VQ_BF16:
        return launch_hadamard_t<__nv_bfloat16, QUANT>(x, diag, n_rows, dim, scale, c, n_c, y, idx, st);
    case VQ_F32: return launch_hadamard_t<float, QUANT>(x, diag, n_rows, dim, scale, c, n_c, y, idx, st);
    }
    return VQ_ERR_INTERNAL;
}

}  // namespace

// fp16 keys against exactly NC (2, 4, 8 or 16) centroids: one block of
// kLookupThreads per SM builds the bucket table once (no workspace).
template <int NC>
vq_status launch_bucket(const void *x, int64_t n, const float *c, uint8_t *out, cudaStream_t st)
{
    const bool vec = (uintptr_t)x % 16 == 0 && (uintptr_t)out % 8 == 0;
    int64_t blocks = (n + 65535) / 65536;  // at least 64 Ki elements per block
    const int sms = vqh_device_sms() > 0 ? vqh_device_sms() : 152;
    if (blocks > sms) blocks = sms;
    if (blocks < 1) blocks = 1;
    auto kp = vqs::scalar_bucket<NC>;
    if (cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, vqs::kBucketSmemBytes) !=
        cudaSuccess)
        return VQ_ERR_CUDA;
    kp<<<(unsigned)blocks, kLookupThreads, vqs::kBucketSmemBytes, st>>>(static_cast<const uint16_t *>(x), n, c,
                                                                        vec, out);
    return launched(st);
}

extern "C" {

size_t vq_scalar_quantize_workspace_bytes(vq_dtype dtype)
{
    return dtype == VQ_F16 || dtype == VQ_BF16 ? kTableBytes : 0;
}

vq_status vq_scalar_quantize(const void *x, vq_dtype dtype, int64_t n, const float *centroids,
                             int32_t n_centroids, uint8_t *out, void *workspace,
                             size_t workspace_bytes, vq_stream_t stream)
{
    if (!dtype_ok(dtype) || n < 0) return VQ_ERR_INVALID_ARG;
    if (n_centroids < 1 || n_centroids > 256) return VQ_ERR_UNSUPPORTED;
    if (n == 0) return VQ_OK;
    if (!x || !centroids || !out) return VQ_ERR_INVALID_ARG;
    if ((uintptr_t)x % elem_size(dtype) || (uintptr_t)centroids % 4) return VQ_ERR_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == VQ_F16) {
        switch (n_centroids) {
        case 2: return launch_bucket<2>(x, n, centroids, out, st);
        case 4: return launch_bucket<4>(x, n, centroids, out, st);
        case 8: return launch_bucket<8>(x, n, centroids, out, st);
        case 16: return launch_bucket<16>(x, n, centroids, out, st);
        }
    }
    const bool table = dtype != VQ_F32 && workspace != nullptr && workspace_bytes >= kTableBytes;
    if (table) {
        if ((uintptr_t)workspace % 16) return VQ_ERR_INVALID_ARG;
        uint8_t *tab = static_cast<uint8_t *>(workspace);
        vqs::scalar_table<<<65536 / kThreads, kThreads, (size_t)n_centroids * 4, st>>>(
            centroids, n_centroids, dtype == VQ_BF16, tab);
        const vq_status ts = launched(st);
        if (ts != VQ_OK) return ts;
        const bool vec = (uintptr_t)x % 16 == 0 && (uintptr_t)out % 8 == 0;
        // one block of kLookupThreads per SM stages the 64 KiB table once;
        // give each block at least 64 Ki elements
        int64_t blocks = (n + 65535) / 65536;
        const int sms = vqh_device_sms() > 0 ? vqh_device_sms() : 152;
        if (blocks > sms) blocks = sms;
        if (blocks < 1) blocks = 1;
        auto kp = vqs::scalar_lookup;
        if (cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTableBytes) !=
            cudaSuccess)
            return VQ_ERR_CUDA;
        kp<<<(unsigned)blocks, kLookupThreads, kTableBytes, st>>>(static_cast<const uint16_t *>(x), n,
                                                                  tab, vec, out);
        return launched(st);
    }
    switch (dtype) {
    case VQ_F16: return launch_scan<__half>(x, n, centroids, n_centroids, out, st);
    case VQ_BF16: return launch_scan<__nv_bfloat16>(x, n, centroids, n_centroids, out, st);
    case VQ_F32: return launch_scan<float>(x, n, centroids, n_centroids, out, st);
    }
    return VQ_ERR_INTERNAL;
}

vq_status vq_scalar_dequantize(const uint8_t *idx, int64_t n, const float *centroids,
                               int32_t n_centroids, vq_dtype dtype, void *out, vq_stream_t stream)
{
    if (!dtype_ok(dtype) || n < 0) return VQ_ERR_INVALID_ARG;
    if (n_centroids < 1 || n_centroids > 256) return VQ_ERR_UNSUPPORTED;
    if (n == 0) return VQ_OK;
    if (!idx || !centroids || !out) return VQ_ERR_INVALID_ARG;
    if ((uintptr_t)centroids % 4 || (uintptr_t)out % elem_size(dtype)) return VQ_ERR_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const unsigned blocks = (unsigned)stream_blocks(n, 8);
    switch (dtype) {
    case VQ_F16:
        vqs::scalar_dequant<__half><<<blocks, kThreads, 0, st>>>(idx, n, centroids, n_centroids,
                                                                 static_cast<__half *>(out));
        break;
    case VQ_BF16:
        vqs::scalar_dequant<__nv_bfloat16><<<blocks, kThreads, 0, st>>>(
            idx, n, centroids, n_centroids, static_cast<__nv_bfloat16 *>(out));
        break;
    case VQ_F32:
        vqs::scalar_dequant<float><<<blocks, kThreads, 0, st>>>(idx, n, centroids, n_centroids,
                                                                static_cast<float *>(out));
        break;
    }
    return launched(st);
}

vq_status vq_hadamard_rotate(const void *x, vq_dtype dtype, const float *diag, int64_t n_rows,
                             int32_t dim, float *y, vq_stream_t stream)
{
    return hadamard<false>(x, dtype, diag, n_rows, dim, nullptr, 0, y, nullptr, stream);
}

vq_status vq_hadamard_quantize(const void *x, vq_dtype dtype, const float *diag, int64_t n_rows,
                               int32_t dim, const float *centroids, int32_t n_centroids,
                               uint8_t *out, vq_stream_t stream)
{
    return hadamard<true>(x, dtype, diag, n_rows, dim, centroids, n_centroids, nullptr, out,
                          stream);
}

}  // extern "C"
