// vq_umma.cuh -- inline-PTX helpers for the 5th-generation tensor cores
// (tcgen05.mma with the accumulator in tensor memory), their shared-memory
// operand descriptors, the mbarrier waits that track them and the
// tensor-memory loads that read the accumulator back, as the encode's
// screening contraction (vq_tc.cuh) uses them.
#pragma once

#include <stdint.h>

namespace vqk {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Shared-memory matrix descriptor: no swizzle, K-major core matrices of
// 8 rows x 16 bytes; lbo = byte distance between core matrices adjacent in K,
// sbo = between core matrices adjacent in M/N.
__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3fff) | ((uint64_t)((lbo >> 4) & 0x3fff) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3fff) << 32) | (1ull << 46);
}

// Instruction descriptor: kind::tf32, fp32 accumulator, A and B K-major,
// M = 128, N = n.
__host__ __device__ constexpr uint32_t umma_idesc_tf32(uint32_t n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// Polls of an mbarrier wait before it gives up.
constexpr int kWaitPolls = 1 << 22;

// Wait for the barrier's phase `parity` to complete, giving up after POLLS
// polls; returns whether it completed.
template <int POLLS = kWaitPolls>
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done = 0;
    for (int it = 0; it < POLLS && !done; ++it) {
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(smem_addr(bar)), "r"(parity)
                     : "memory");
    }
    return done != 0;
}

// Bits of a thread's wait state.
constexpr uint32_t kWaitLate = 1u;    // a wait completed only after more than POLLS polls, or not at all
constexpr uint32_t kWaitFailed = 2u;  // a wait did not complete within the full limit

// Wait for the barrier's phase `parity` to complete, polling up to the full
// limit whatever POLLS is, and classify the wait: 0 if it completed within
// POLLS polls, kWaitLate if it completed later, kWaitLate | kWaitFailed if
// it did not complete.  With POLLS equal to the full limit this is mbar_wait.
template <int POLLS>
__device__ __forceinline__ uint32_t mbar_wait_state(uint64_t *bar, uint32_t parity)
{
    uint32_t done = 0;
    int it = 0;
    for (; it < kWaitPolls && !done; ++it) {
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(smem_addr(bar)), "r"(parity)
                     : "memory");
    }
    if (!done) return kWaitLate | kWaitFailed;
    if constexpr (POLLS < kWaitPolls) return it > POLLS ? kWaitLate : 0u;
    return 0u;
}

// Arrive once on the barrier (completing a phase of arrival count 1);
// returns the barrier state token, which callers may ignore.
__device__ __forceinline__ uint64_t mbar_arrive(uint64_t *bar)
{
    uint64_t state;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(state) : "r"(smem_addr(bar)) : "memory");
    return state;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns, without waiting: the registers are valid only
// after tmem_wait_ld.
__device__ __forceinline__ void tmem_load32_async(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Wait for this thread's outstanding tensor-memory loads.  The empty
// statements make every loaded register an output of the wait, so no use of
// one can be scheduled above it.
template <int N>
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[N])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < N; ++j) asm volatile("" : "+r"(r[j]));
}

}  // namespace vqk
