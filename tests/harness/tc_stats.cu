// tc_stats.cu -- test-only: the library's tensor-core encode (vq_tc.cuh) in
// its library configuration (vqk::TcConfig, full poll limit), compiled with
// VQ_TC_STATS so that every encoded row also counts its screening outcome:
// one candidate group, two, or the exact queue, each split by whether the
// least excluded group minimum lay within one bound of the threshold.  The
// indices are the library's.  Built by the tests; not part of libvqenc.so.
#define VQ_TC_STATS 1

#include <cuda_runtime.h>

#include <type_traits>

#include "vq_tc.cuh"

namespace {

template <typename T, int SUB, bool SMOOTH>
cudaError_t launch(const void *x, const void *cb, int64_t n_groups, int64_t n_per_group,
                   int32_t n_c, int32_t tiles_per_block, uint32_t *out, const float *smooth,
                   int32_t head_dim, cudaStream_t st)
{
    constexpr bool kF32 = std::is_same<T, float>::value;
    using C = vqk::TcConfig<SUB, SMOOTH || kF32>;
    using L = vqk::TcLayout<SUB, C::kCols, C::kGroup, SMOOTH || kF32 ? 2 : 1, kF32 ? 2 : 1, C::kTps>;
    const size_t smem = L::bytes(n_c);
    auto k = vqk::encode_tc<T, SUB, C::kCols, C::kGroup, C::kMinBlocks, uint32_t, SMOOTH, vqk::kWaitPolls, C::kTps>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (n_per_group + 127) / 128;
    const int64_t per_group = (tiles + tiles_per_block - 1) / tiles_per_block;
    k<<<(unsigned)(n_groups * per_group), 128 * C::kTps, smem, st>>>(
        static_cast<const T *>(x), static_cast<const T *>(cb), n_per_group, n_c, per_group,
        tiles_per_block, 1.0f, out, smooth, SMOOTH ? head_dim / SUB : 1);
    return cudaPeekAtLastError();
}

template <typename T>
cudaError_t launch_sub(int sub, int smooth, const void *x, const void *cb, int64_t g, int64_t m,
                       int32_t n_c, int32_t t, uint32_t *out, const float *s, int32_t hd,
                       cudaStream_t st)
{
    if (sub == 4) return smooth ? launch<T, 4, true>(x, cb, g, m, n_c, t, out, s, hd, st)
                                : launch<T, 4, false>(x, cb, g, m, n_c, t, out, s, hd, st);
    if (sub == 8) return smooth ? launch<T, 8, true>(x, cb, g, m, n_c, t, out, s, hd, st)
                                : launch<T, 8, false>(x, cb, g, m, n_c, t, out, s, hd, st);
    return cudaErrorInvalidValue;
}

}  // namespace

// The library's grouped encode with statistics.  dtype 0 fp16, 1 bf16, 2 fp32;
// sub 4 or 8; 64 <= n_c <= 256; x aligned to its row; smooth != 0 takes the
// factors [n_groups][head_dim] (n_per_group a multiple of head_dim / sub).
extern "C" int stats_encode(int dtype, int sub, int smooth, const void *x, const void *cb,
                            int64_t n_groups, int64_t n_per_group, int32_t n_c,
                            int32_t tiles_per_block, uint32_t *out, const float *factors,
                            int32_t head_dim, cudaStream_t st)
{
    if (n_groups < 1 || n_per_group < 1 || n_c < 64 || n_c > 256 || tiles_per_block < 1 ||
        (smooth && (head_dim < sub || head_dim % sub || n_per_group % (head_dim / sub))))
        return (int)cudaErrorInvalidValue;
    switch (dtype) {
    case 0: return (int)launch_sub<__half>(sub, smooth, x, cb, n_groups, n_per_group, n_c, tiles_per_block, out, factors, head_dim, st);
    case 1: return (int)launch_sub<__nv_bfloat16>(sub, smooth, x, cb, n_groups, n_per_group, n_c, tiles_per_block, out, factors, head_dim, st);
    case 2: return (int)launch_sub<float>(sub, smooth, x, cb, n_groups, n_per_group, n_c, tiles_per_block, out, factors, head_dim, st);
    }
    return (int)cudaErrorInvalidValue;
}

// Read (after a device synchronisation) and optionally clear the counters:
// out[0..4] = rows with 1 candidate group, 1 (tight), 2, 2 (tight), queued.
extern "C" int stats_read(unsigned long long *out, int clear)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(out, vqk::g_tc_stats, 8 * sizeof(unsigned long long));
    if (e == cudaSuccess && clear) {
        const unsigned long long zero[8] = {};
        e = cudaMemcpyToSymbol(vqk::g_tc_stats, zero, sizeof zero);
    }
    return (int)e;
}

// This unit's device status word (vq_status.cuh), optionally cleared.
extern "C" int stats_status(uint32_t *bits, int clear)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, vqk::g_status_word, sizeof(uint32_t));
    if (e == cudaSuccess && clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(vqk::g_status_word, &zero, sizeof zero);
    }
    return (int)e;
}
