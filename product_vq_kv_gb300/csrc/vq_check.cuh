// vq_check.cuh -- the bounds checks of the checked build.
//
// Compiled with -DVQ_CHECKED (libvqenc_checked.so), every index that the
// encode, attention, scalar and Hadamard kernels compute into a global or a
// shared buffer is checked before the access: the span must lie inside the
// buffer it belongs to and be aligned for its access width.  A span outside
// sets kStatusOutOfBounds in the device status word (vq_status.cuh) and the
// access is skipped (a skipped load leaves its value zero); nothing traps.
// The entry points of the checked library synchronise after their launches
// and turn the bit into VQ_ERR_INTERNAL.  This stands in for a memory
// checker on machines where none may run.
//
// In the library build kChecked is false: every check is the constant true
// and compiles away, and the kernels are the ones measured.
#pragma once

#include <stdint.h>

#include "vq_status.cuh"

namespace vqk {

#ifdef VQ_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// Does the span [p, p + bytes) lie inside [base, base + region) and start at
// a multiple of `align` (the width of the accesses that will be made)?
// Generic addresses: shared or global.
__device__ __forceinline__ bool span_ok(const void *p, uint64_t bytes, const void *base,
                                        uint64_t region, uint32_t align)
{
    if constexpr (!kChecked) {
        return true;
    } else {
        const uint64_t a = (uint64_t)(uintptr_t)p, b = (uint64_t)(uintptr_t)base;
        if (a >= b && a - b <= region && bytes <= region - (a - b) && a % align == 0) return true;
        raise_status(kStatusOutOfBounds);
        return false;
    }
}

// Is `index` inside [0, n)?  For register arrays, tensor-memory columns and
// similar indices that are not addresses.
__device__ __forceinline__ bool index_ok(int64_t index, int64_t n)
{
    if constexpr (!kChecked) {
        return true;
    } else {
        if (index >= 0 && index < n) return true;
        raise_status(kStatusOutOfBounds);
        return false;
    }
}

// Does the span [p, p + bytes) lie inside this launch's dynamic shared
// memory, starting at a multiple of `align`?
__device__ __forceinline__ bool dyn_smem_ok(const void *p, uint64_t bytes, uint32_t align)
{
    if constexpr (!kChecked) {
        return true;
    } else {
        extern __shared__ unsigned char vq_check_dyn_smem[];
        uint32_t size;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
        return span_ok(p, bytes, vq_check_dyn_smem, size, align);
    }
}

}  // namespace vqk

// A span of `count` elements at `ptr` inside the buffer of `n` elements at
// `base` (both counted in the element type of `ptr`), accessed element by
// element (aligned to the element size, at most 16 bytes).
#define VQ_SPAN(ptr, count, base, n)                                                        \
    (::vqk::span_ok((ptr), (uint64_t)(count) * sizeof(*(ptr)), (base),                    \
                    (uint64_t)(n) * sizeof(*(ptr)), sizeof(*(ptr)) < 16 ? sizeof(*(ptr)) : 16))
// The same span accessed with vector loads or stores of `vec` bytes.
#define VQ_VSPAN(ptr, count, base, n, vec)                                                  \
    (::vqk::span_ok((ptr), (uint64_t)(count) * sizeof(*(ptr)), (base),                    \
                    (uint64_t)(n) * sizeof(*(ptr)), (vec)))
