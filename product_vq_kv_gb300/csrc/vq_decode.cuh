// vq_decode.cuh -- product-VQ decode ("dequantize_vq"): indices back to
// sub-vectors, out[g][m][:] = codebooks[g][idx[g][m]][:], an exact copy of
// the codebook row (source: "I Wrote a Metal Kernel to Stop My Mac From
// OOMing", section "Mistake 1: I Wrote the Dequant Kernel First" -- the
// operation that takes codebook indices and reconstructs the vectors, a
// gather).  An index outside [0, n_centroids) gives a row of zeros.
//
// The work is a byte gather bound by HBM bandwidth: per row the index (1 or
// 4 bytes) is read and the row (sub_dim elements) written; the codebook (a
// few KiB per group) stays in the L1 / read-only cache.  Rows move as 8-,
// 16- or 32-byte vectors; indices are read and rows written coalesced (thread
// t of a block handles rows t, t + THREADS, ...), with streaming stores.
#pragma once

#include <stdint.h>

namespace vqk {

template <int BYTES>
struct RowVec;
template <>
struct RowVec<8> {
    uint2 a;
};
template <>
struct RowVec<16> {
    uint4 a;
};
template <>
struct RowVec<32> {
    uint4 a, b;
};

template <int BYTES>
__device__ __forceinline__ RowVec<BYTES> load_cb_row(const unsigned char *p)
{
    RowVec<BYTES> v;
    if constexpr (BYTES == 8) {
        v.a = __ldg(reinterpret_cast<const uint2 *>(p));
    } else if constexpr (BYTES == 16) {
        v.a = __ldg(reinterpret_cast<const uint4 *>(p));
    } else {
        v.a = __ldg(reinterpret_cast<const uint4 *>(p));
        v.b = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
    }
    return v;
}

template <int BYTES>
__device__ __forceinline__ RowVec<BYTES> zero_row()
{
    RowVec<BYTES> v;
    if constexpr (BYTES == 8) {
        v.a = make_uint2(0, 0);
    } else if constexpr (BYTES == 16) {
        v.a = make_uint4(0, 0, 0, 0);
    } else {
        v.a = make_uint4(0, 0, 0, 0);
        v.b = make_uint4(0, 0, 0, 0);
    }
    return v;
}

template <int BYTES>
__device__ __forceinline__ void store_row(unsigned char *p, const RowVec<BYTES> &v)
{
    if constexpr (BYTES == 8) {
        __stcs(reinterpret_cast<uint2 *>(p), v.a);
    } else if constexpr (BYTES == 16) {
        __stcs(reinterpret_cast<uint4 *>(p), v.a);
    } else {
        __stcs(reinterpret_cast<uint4 *>(p), v.a);
        __stcs(reinterpret_cast<uint4 *>(p) + 1, v.b);
    }
}

__device__ __forceinline__ uint32_t load_index(const uint32_t *p) { return __ldcs(p); }
__device__ __forceinline__ uint32_t load_index(const uint8_t *p) { return *p; }

// Launch: grid.x = n_groups * blocks_per_group, block = THREADS; block b
// decodes rows [(b % blocks_per_group) * THREADS * R, ...) of group
// b / blocks_per_group.  Requires codebooks and out aligned to
// min(ROW_BYTES, 16) bytes.
template <typename IdxT, int ROW_BYTES, int THREADS, int R>
__global__ void __launch_bounds__(THREADS)
    decode_rows(const IdxT *__restrict__ idx, const unsigned char *__restrict__ codebooks,
                int64_t n_per_group, int32_t n_centroids, int64_t blocks_per_group,
                unsigned char *__restrict__ out)
{
    const int64_t g = blockIdx.x / blocks_per_group;
    const int64_t blk = blockIdx.x - g * blocks_per_group;
    const unsigned char *__restrict__ cb = codebooks + (size_t)g * (size_t)n_centroids * ROW_BYTES;
    const IdxT *__restrict__ ig = idx + (size_t)g * (size_t)n_per_group;
    unsigned char *__restrict__ og = out + (size_t)g * (size_t)n_per_group * ROW_BYTES;
    const int64_t row0 = blk * (int64_t)(THREADS * R) + threadIdx.x;
    uint32_t k[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + (int64_t)r * THREADS;
        k[r] = row < n_per_group ? load_index(ig + row) : 0u;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + (int64_t)r * THREADS;
        if (row < n_per_group) {
            const RowVec<ROW_BYTES> v = k[r] < (uint32_t)n_centroids
                                            ? load_cb_row<ROW_BYTES>(cb + (size_t)k[r] * ROW_BYTES)
                                            : zero_row<ROW_BYTES>();
            store_row<ROW_BYTES>(og + (size_t)row * ROW_BYTES, v);
        }
    }
}

// Any row size and alignment (elements of ELEM bytes): one thread per output
// element.  Launch: grid.x = ceil(n_groups * n_per_group * sub_dim / blockDim.x).
template <typename IdxT, typename ElemT>
__global__ void decode_elems(const IdxT *__restrict__ idx, const ElemT *__restrict__ codebooks,
                             int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                             int32_t sub_dim, ElemT *__restrict__ out)
{
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = n_groups * n_per_group * sub_dim;
    if (e >= total) return;
    const int64_t row = e / sub_dim;
    const int32_t i = (int32_t)(e - row * sub_dim);
    const int64_t g = row / n_per_group;
    const uint32_t k = load_index(idx + row);
    ElemT v{};
    if (k < (uint32_t)n_centroids)
        v = codebooks[((size_t)g * (size_t)n_centroids + k) * (size_t)sub_dim + i];
    out[e] = v;
}

}  // namespace vqk
