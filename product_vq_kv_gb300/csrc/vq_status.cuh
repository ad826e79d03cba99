// vq_status.cuh -- the device status word: bits a kernel sets when it could
// not finish its work normally, read back on the host by vq_kernel_status().
//
// The word is a file-scope `static __device__` variable, so every translation
// unit that includes this header (and every device it runs on) has its own
// copy; each .cu file of the library exports a host function that reads and
// clears its copy (vq_host.h), and vq_kernel_status() ORs them.  Kernels only
// ever OR bits in (atomicOr), never trap, and keep running or return.
#pragma once

#include <stdint.h>

namespace vqk {

// A tensor-core wait gave up: the block's unfinished rows hold the marker
// 0xFFFFFFFF (0xFF as 8-bit codes).
constexpr uint32_t kStatusWaitGaveUp = 1u;
// Bounds-checked build only: an index fell outside its buffer and the access
// was skipped.
constexpr uint32_t kStatusOutOfBounds = 2u;

static __device__ uint32_t g_status_word;

__device__ __forceinline__ void raise_status(uint32_t bits) { atomicOr(&g_status_word, bits); }

}  // namespace vqk
