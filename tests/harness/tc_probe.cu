// tc_probe.cu -- test-only kernel: one chain of tcgen05.mma kind::tf32 per
// 128-row tile, issued through the same shared-memory descriptors,
// instruction descriptor, commit, bounded mbarrier wait and tensor-memory
// loads as the library's tensor-core encode (vq_tc.cuh), so that the GPU
// tests can measure the accumulation error of exactly those products.
// Built by the tests (tests/tc_harness.py); not part of libvqenc.so.
//
//   A  [ntiles][128][8 NK]     fp32 holding tf32 values (row-major)
//   B  [ntiles][NCOLS][8 NK]   fp32 holding tf32 values
//   D  [ntiles][128][NCOLS]    fp32, written: D = sum over the NK K-steps of
//                              the 128 x 8 by 8 x NCOLS products, accumulated
//                              in tensor memory (the first step overwrites)
//   flag                       bit 0 set if a wait gave up (D not written)
#include <cuda_runtime.h>

#include "vq_tc.cuh"

namespace {

template <int NK, int NCOLS>
struct ProbeLayout {
    static constexpr int kK = 8 * NK;   // tf32 elements per row
    static constexpr int kKB = kK / 4;  // 16-byte core-matrix columns per row
    static constexpr size_t kA = (size_t)128 * kK * 4;
    static constexpr size_t kB = (size_t)NCOLS * kK * 4;
    static constexpr size_t kUsed = kA + kB + 16 + 1024;  // barrier, slot, 1 KiB alignment
    // at least 1 / (512 / NCOLS + 1) of an SM's 228 KiB, so the resident CTAs
    // never ask for more than its 512 tensor-memory columns
    static constexpr size_t kCap = (size_t)228 * 1024 / (512 / NCOLS + 1) + 1024;
    static constexpr size_t kBytes = kUsed > kCap ? kUsed : kCap;
};

template <int NK, int NCOLS>
__global__ void __launch_bounds__(128, 1)
    tf32_chain(const float *__restrict__ A, const float *__restrict__ B, float *__restrict__ D,
               uint32_t *__restrict__ flag)
{
    using L = ProbeLayout<NK, NCOLS>;
    extern __shared__ unsigned char raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    float *sa = reinterpret_cast<float *>(sm);
    float *sb = reinterpret_cast<float *>(sm + L::kA);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::kA + L::kB);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5;
    const size_t tile = blockIdx.x;
    const float *At = A + tile * 128 * L::kK;
    const float *Bt = B + tile * NCOLS * L::kK;

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(vqk::smem_addr(bar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         vqk::smem_addr(tslot)),
                     "r"(NCOLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // K-major core matrices of 8 rows x 16 bytes, as encode_tc lays them out
    for (int kb = 0; kb < L::kKB; ++kb)
        *reinterpret_cast<float4 *>(sa + ((tid >> 3) * (L::kKB * 128) + kb * 128 + (tid & 7) * 16) / 4) =
            *reinterpret_cast<const float4 *>(At + (size_t)tid * L::kK + 4 * kb);
    for (int c = tid; c < NCOLS; c += 128)
        for (int kb = 0; kb < L::kKB; ++kb)
            *reinterpret_cast<float4 *>(sb + ((c >> 3) * (L::kKB * 128) + kb * 128 + (c & 7) * 16) / 4) =
                *reinterpret_cast<const float4 *>(Bt + (size_t)c * L::kK + 4 * kb);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    vqk::tc_fence_before();
    __syncthreads();
    vqk::tc_fence_after();
    const uint32_t tmem = *tslot;

    if (tid == 0) {
        const uint32_t idesc = vqk::umma_idesc_tf32((uint32_t)NCOLS);
        constexpr uint32_t kSbo = L::kKB * 128;
        for (int ks = 0; ks < NK; ++ks)
            vqk::umma_tf32(tmem, vqk::umma_smem_desc(vqk::smem_addr(sa) + ks * 256, 128, kSbo),
                           vqk::umma_smem_desc(vqk::smem_addr(sb) + ks * 256, 128, kSbo), idesc,
                           ks > 0);
        vqk::umma_commit(bar);
    }
    const bool done = vqk::mbar_wait(bar, 0);
    vqk::tc_fence_after();
    if (__all_sync(0xffffffffu, done)) {
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        float *Dt = D + tile * 128 * NCOLS + (size_t)tid * NCOLS;
        for (int j = 0; j < NCOLS; j += 32) {
            uint32_t v[32];
            vqk::tmem_load32_async(tmem + lane_base + (uint32_t)j, v);
            vqk::tmem_wait_ld(v);
#pragma unroll
            for (int q = 0; q < 32; q += 4)
                *reinterpret_cast<float4 *>(Dt + j + q) =
                    make_float4(__uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
        }
    } else if ((tid & 31) == 0) {
        atomicOr(flag, 1u);
    }
    vqk::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // a wait that gave up: thread 0 (which issued the only MMA chain)
        // waits once more, with the full limit, before the memory is freed
        if (tid == 0 && !done) (void)vqk::mbar_wait(bar, 0);
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NCOLS));
    }
}

template <int NK, int NCOLS>
cudaError_t launch(const float *A, const float *B, float *D, uint32_t *flag, int ntiles,
                   cudaStream_t st)
{
    auto k = tf32_chain<NK, NCOLS>;
    const size_t smem = ProbeLayout<NK, NCOLS>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<(unsigned)ntiles, 128, smem, st>>>(A, B, D, flag);
    return cudaPeekAtLastError();
}

template <int NK>
cudaError_t launch_cols(int ncols, const float *A, const float *B, float *D, uint32_t *flag,
                        int ntiles, cudaStream_t st)
{
    switch (ncols) {
    case 64: return launch<NK, 64>(A, B, D, flag, ntiles, st);
    case 256: return launch<NK, 256>(A, B, D, flag, ntiles, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

// D = A B^T per tile (see the header of this file); nk in {1, 2, 3, 4, 6},
// ncols in {64, 256}, ntiles >= 1.  Returns a cudaError_t code.
extern "C" int probe_tf32_chain(const float *A, const float *B, float *D, uint32_t *flag, int nk,
                                int ncols, int ntiles, cudaStream_t st)
{
    if (ntiles < 1 || !A || !B || !D || !flag) return (int)cudaErrorInvalidValue;
    switch (nk) {
    case 1: return (int)launch_cols<1>(ncols, A, B, D, flag, ntiles, st);
    case 2: return (int)launch_cols<2>(ncols, A, B, D, flag, ntiles, st);
    case 3: return (int)launch_cols<3>(ncols, A, B, D, flag, ntiles, st);
    case 4: return (int)launch_cols<4>(ncols, A, B, D, flag, ntiles, st);
    case 6: return (int)launch_cols<6>(ncols, A, B, D, flag, ntiles, st);
    }
    return (int)cudaErrorInvalidValue;
}
