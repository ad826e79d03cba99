// tc_polls.cu -- test-only: the library's tensor-core encode (vq_tc.cuh) in
// its library configuration except for the per-pass poll limit of its
// mbarrier waits, which is tiny here (0 or 1 polls), so that the waits give
// up while every MMA still completes: the path that marks unfinished rows,
// records kStatusWaitGaveUp and frees tensor memory only after the last MMA
// it issued.  The cleanup wait keeps the full limit.  Built by the tests; not
// part of libvqenc.so.
#include <cuda_runtime.h>

#include "vq_tc.cuh"

namespace {

template <int POLLS, int SUB, typename OutT>
cudaError_t launch(const void *x, const void *cb, int64_t n_groups, int64_t n_per_group,
                   int32_t n_c, int32_t tiles_per_block, void *out, cudaStream_t st)
{
    using C = vqk::TcConfig<SUB>;
    using L = vqk::TcLayout<SUB, C::kCols, C::kGroup, 1, 1, C::kTps>;
    const size_t smem = L::bytes(n_c);
    auto k = vqk::encode_tc<__half, SUB, C::kCols, C::kGroup, C::kMinBlocks, OutT, false, POLLS, C::kTps>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (n_per_group + 127) / 128;
    const int64_t per_group = (tiles + tiles_per_block - 1) / tiles_per_block;
    k<<<(unsigned)(n_groups * per_group), 128 * C::kTps, smem, st>>>(
        static_cast<const __half *>(x), static_cast<const __half *>(cb), n_per_group, n_c,
        per_group, tiles_per_block, 1.0f, static_cast<OutT *>(out), nullptr, 1);
    return cudaPeekAtLastError();
}

template <int POLLS>
cudaError_t launch_polls(int sub, int out_bytes, const void *x, const void *cb, int64_t g,
                         int64_t m, int32_t n_c, int32_t t, void *out, cudaStream_t st)
{
    if (sub == 4 && out_bytes == 4) return launch<POLLS, 4, uint32_t>(x, cb, g, m, n_c, t, out, st);
    if (sub == 4 && out_bytes == 1) return launch<POLLS, 4, uint8_t>(x, cb, g, m, n_c, t, out, st);
    if (sub == 8 && out_bytes == 4) return launch<POLLS, 8, uint32_t>(x, cb, g, m, n_c, t, out, st);
    return cudaErrorInvalidValue;
}

}  // namespace

// fp16 grouped encode with `polls` (0 or 1) polls per wait; sub 4 (uint32 or
// uint8 out) or 8 (uint32); 64 <= n_c <= 256; x aligned to its row.
extern "C" int polls_encode(int polls, int sub, int out_bytes, const void *x, const void *cb,
                            int64_t n_groups, int64_t n_per_group, int32_t n_c,
                            int32_t tiles_per_block, void *out, cudaStream_t st)
{
    if (n_groups < 1 || n_per_group < 1 || n_c < 64 || n_c > 256 || tiles_per_block < 1)
        return (int)cudaErrorInvalidValue;
    if (polls == 0) return (int)launch_polls<0>(sub, out_bytes, x, cb, n_groups, n_per_group, n_c, tiles_per_block, out, st);
    if (polls == 1) return (int)launch_polls<1>(sub, out_bytes, x, cb, n_groups, n_per_group, n_c, tiles_per_block, out, st);
    return (int)cudaErrorInvalidValue;
}

// This unit's device status word (vq_status.cuh), optionally cleared.
extern "C" int polls_status(uint32_t *bits, int clear)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, vqk::g_status_word, sizeof(uint32_t));
    if (e == cudaSuccess && clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(vqk::g_status_word, &zero, sizeof zero);
    }
    return (int)e;
}
