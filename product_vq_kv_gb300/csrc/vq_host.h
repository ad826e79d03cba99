// vq_host.h -- host helpers shared by the library's translation units
// (internal; not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "vq_encode.h"

// Streaming multiprocessors of the current device, cached per device; 0 if
// there is no usable device.
int vqh_device_sms();

// OR into *bits this translation unit's device status word on the current
// device (vq_status.cuh), then reset it to zero if `clear`.  The caller has
// synchronised the device.
cudaError_t vqh_status_encode(uint32_t *bits, bool clear);
cudaError_t vqh_status_attn(uint32_t *bits, bool clear);
cudaError_t vqh_status_scalar(uint32_t *bits, bool clear);

// The body of the three functions above, for the translation unit's own word.
#define VQH_STATUS_READER(NAME)                                                      \
    cudaError_t NAME(uint32_t *bits, bool clear)                                     \
    {                                                                                \
        uint32_t v = 0;                                                              \
        cudaError_t e = cudaMemcpyFromSymbol(&v, vqk::g_status_word, sizeof v);      \
        if (e != cudaSuccess) return e;                                              \
        *bits |= v;                                                                  \
        if (clear && v != 0) {                                                       \
            const uint32_t zero = 0;                                                 \
            e = cudaMemcpyToSymbol(vqk::g_status_word, &zero, sizeof zero);          \
        }                                                                            \
        return e;                                                                    \
    }

// Status of the launches just made on `stream`: VQ_ERR_CUDA if a launch
// failed, else VQ_OK.  In the checked build (VQ_CHECKED) the call also waits
// for them and reports an out-of-bounds bit in this unit's status word (read
// by `reader`) as VQ_ERR_INTERNAL; the bit stays set until vq_kernel_status()
// clears it.
inline vq_status vqh_launched(cudaStream_t stream, cudaError_t (*reader)(uint32_t *, bool))
{
    if (cudaPeekAtLastError() != cudaSuccess) return VQ_ERR_CUDA;
#ifdef VQ_CHECKED
    if (cudaStreamSynchronize(stream) != cudaSuccess) return VQ_ERR_CUDA;
    uint32_t bits = 0;
    if (reader(&bits, false) != cudaSuccess) return VQ_ERR_CUDA;
    if (bits & VQ_KSTATUS_OUT_OF_BOUNDS) return VQ_ERR_INTERNAL;
#else
    (void)stream;
    (void)reader;
#endif
    return VQ_OK;
}
