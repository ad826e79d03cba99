// link_probe.cu -- test-only kernel: reads a buffer 16 bytes per thread, four
// loads in flight per thread, and writes the XOR of the two halves of each
// 16 bytes as 8 bytes, so that a GPU test can measure the rate at which the
// SMs read pinned host memory across the CPU-GPU link, beside the
// host-buffer encode, which reads its input the same way (vq_encode.h,
// vq_encode_grouped_host).  Built by the tests (tests/tc_harness.py); not
// part of libvqenc.so.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__global__ void link_read(const uint4 *__restrict__ x, int64_t n, uint2 *__restrict__ out)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldcs(x + i + k * stride);
#pragma unroll
        for (int k = 0; k < 4; ++k) __stcs(out + i + k * stride, make_uint2(v[k].x ^ v[k].z, v[k].y ^ v[k].w));
    }
    for (; i < n; i += stride) {
        const uint4 v = __ldcs(x + i);
        __stcs(out + i, make_uint2(v.x ^ v.z, v.y ^ v.w));
    }
}

}  // namespace

// x: `bytes` (a multiple of 16) device or pinned host bytes, 16-byte aligned;
// out: bytes / 2 device bytes.  Returns a cudaError_t code.
extern "C" int probe_link_read(const void *x, int64_t bytes, void *out, int blocks, cudaStream_t st)
{
    if (!x || !out || bytes <= 0 || bytes % 16 || blocks < 1 || ((uintptr_t)x & 15u) || ((uintptr_t)out & 7u))
        return (int)cudaErrorInvalidValue;
    link_read<<<blocks, 256, 0, st>>>(static_cast<const uint4 *>(x), bytes / 16, static_cast<uint2 *>(out));
    return (int)cudaPeekAtLastError();
}
