// check_probe.cu -- test-only: evaluates the checked build's bounds-check
// primitives (vq_check.cuh) on spans the host describes, without reading or
// writing the memory they describe, so that the GPU tests can pin what the
// checks accept and reject.  Built by the tests; not part of libvqenc.so.
#define VQ_CHECKED 1

#include <cuda_runtime.h>

#include "vq_check.cuh"

namespace {

// One block of n threads (n <= 1024) with `smem` bytes of dynamic shared
// memory; thread k evaluates case k and writes 1 (accepted) or 0:
//   kind 0: dyn_smem_ok(shared + off, bytes, align)
//   kind 1: span_ok(gbase + off, bytes, gbase, region, align)   (gbase: any
//           global address; nothing is dereferenced)
// with align = the largest of 16, 8, 4, 2, 1 not above bytes
//   kind 2: index_ok(off, region)
__global__ void check_cases(const int *__restrict__ kind, const long long *__restrict__ off,
                            const long long *__restrict__ bytes,
                            const long long *__restrict__ region, int n,
                            const unsigned char *gbase, int *__restrict__ result)
{
    extern __shared__ unsigned char probe_smem[];
    const int k = threadIdx.x;
    if (k >= n) return;
    bool ok = false;
    // the access width a span of this many bytes would be made with
    const uint32_t align = bytes[k] >= 16 ? 16 : bytes[k] >= 8 ? 8 : bytes[k] >= 4 ? 4 : bytes[k] >= 2 ? 2 : 1;
    switch (kind[k]) {
    case 0: ok = vqk::dyn_smem_ok(probe_smem + off[k], (uint64_t)bytes[k], align); break;
    case 1: ok = vqk::span_ok(gbase + off[k], (uint64_t)bytes[k], gbase, (uint64_t)region[k], align); break;
    case 2: ok = vqk::index_ok(off[k], region[k]); break;
    }
    result[k] = ok ? 1 : 0;
}

}  // namespace

extern "C" int check_probe(const int *kind, const long long *off, const long long *bytes,
                           const long long *region, int n, const void *gbase, int *result,
                           int smem_bytes, cudaStream_t st)
{
    if (n < 1 || n > 1024 || smem_bytes < 0 || smem_bytes > 48 * 1024) return (int)cudaErrorInvalidValue;
    check_cases<<<1, n, (size_t)smem_bytes, st>>>(kind, off, bytes, region, n,
                                                  static_cast<const unsigned char *>(gbase), result);
    return (int)cudaPeekAtLastError();
}

// This unit's device status word, optionally cleared.
extern "C" int check_status(uint32_t *bits, int clear)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(bits, vqk::g_status_word, sizeof(uint32_t));
    if (e == cudaSuccess && clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(vqk::g_status_word, &zero, sizeof zero);
    }
    return (int)e;
}
