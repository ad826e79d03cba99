// vq_kernels.cuh -- sm_103a kernels for product-VQ encode (nearest centroid).
//
// What is computed (from "I Wrote a Metal Kernel to Stop My Mac From
// OOMing", section "The Kernel: 18 Lines of MSL"): for every sub-vector x of
// length SUB, dist(c) = sum_i (float(x_i) - float(c_i))^2 in fp32, each
// subtract, square and add rounded separately, summed in ascending i; the
// index written is the smallest c with the least dist (strict "<" running
// argmin from (+inf, 0); NaN never wins).  The kernels reproduce that
// definition bit for bit.
//
// GB300 design (the page's shader -- one thread per sub-vector, codebook read
// from device memory on every centroid -- is prior art, not the plan):
//  * The codebook of the block's group is staged once per block into shared
//    memory, widened to fp32 and negated, each value stored twice
//    (-c_i, -c_i).  Reads in the centroid loop are warp-uniform broadcasts.
//  * Each thread owns R sub-vectors, held in registers as R/2 packed pairs.
//    One packed f32x2 add / multiply evaluates the same centroid against two
//    sub-vectors at once; each lane rounds exactly like the scalar fp32 op
//    (see "Exact fp32 arithmetic" below for how contraction into an FMA is
//    ruled out), so the result is bit-identical.  Packed ops issue at half the rate of scalar
//    ones (same FP32 lane throughput) but halve the issue slots taken, which
//    leaves room for the argmin's compare/select work on the ALU pipe.
//  * x is read with 8/16-byte vector loads in a coalesced pattern (thread t
//    of a block owns rows t, t+THREADS, ...); indices leave with coalesced
//    32-bit streaming stores.  Nothing but x, the codebooks and the indices
//    touches device memory.
//  * Two argmin strategies (template MODE):
//      kDirect   : per centroid, compare-and-select (dist, index) per row.
//      kDeferred : per pair of centroids one three-input fp32 min keeps the
//                  running minimum; per group of GC centroids one compare
//                  remembers the first group that lowered it; at the end the
//                  winning group alone is re-evaluated to find the first
//                  centroid whose distance equals the minimum.  Same result:
//                  the minimum is one of the exactly computed distances, the
//                  first group that reaches it holds its lowest index, and
//                  re-evaluation reproduces the distances bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace vqk {

enum ArgminMode { kDirect = 0, kDeferred = 1 };

// ------------------------------------------------------------------ element types

__device__ __forceinline__ float widen(__half v) { return __half2float(v); }
__device__ __forceinline__ float widen(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float widen(float v) { return v; }

template <typename T>
__device__ __forceinline__ T from_bits(unsigned short u);
template <>
__device__ __forceinline__ __half from_bits<__half>(unsigned short u) { return __ushort_as_half(u); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_bits<__nv_bfloat16>(unsigned short u)
{
    return __ushort_as_bfloat16(u);
}

// Load one row of SUB elements (SUB * sizeof(T) bytes, aligned to that size or
// to 16 bytes, whichever is smaller) with vector loads and widen it to fp32.
template <typename T, int SUB>
__device__ __forceinline__ void load_row(const T *__restrict__ p, float (&v)[SUB])
{
    constexpr int kBytes = SUB * (int)sizeof(T);
    static_assert(kBytes % 8 == 0, "rows must be a multiple of 8 bytes");
    uint32_t w[kBytes / 4];
    if constexpr (kBytes % 16 == 0) {
#pragma unroll
        for (int k = 0; k < kBytes / 16; ++k) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(p) + k);
            w[4 * k + 0] = q.x;
            w[4 * k + 1] = q.y;
            w[4 * k + 2] = q.z;
            w[4 * k + 3] = q.w;
        }
    } else {
        const uint2 q = __ldcs(reinterpret_cast<const uint2 *>(p));
        w[0] = q.x;
        w[1] = q.y;
    }
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < SUB; ++i) v[i] = __uint_as_float(w[i]);
    } else {
#pragma unroll
        for (int j = 0; j < SUB / 2; ++j) {
            const T lo = from_bits<T>(static_cast<unsigned short>(w[j] & 0xffffu));
            const T hi = from_bits<T>(static_cast<unsigned short>(w[j] >> 16));
            v[2 * j] = widen(lo);
            v[2 * j + 1] = widen(hi);
        }
    }
}

// Store one index: uint32 (streaming store) or uint8 codes.
__device__ __forceinline__ void store_index(uint32_t *p, uint32_t v) { __stcs(p, v); }
__device__ __forceinline__ void store_index(uint8_t *p, uint32_t v) { *p = (uint8_t)v; }

// ------------------------------------------------------------------ arithmetic

// Three-input fp32 minimum (sm_100+).  NaN inputs are ignored unless all are
// NaN, so a NaN distance never lowers the running minimum.
__device__ __forceinline__ float min3(float a, float b, float c)
{
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Exact fp32 arithmetic.
//
// The distance needs the square and the running sum rounded separately.
// ptxas contracts a packed mul.rn.f32x2 whose only use is an add.rn.f32x2
// into one fused multiply-add, whatever the rounding modifiers and the -fmad
// setting say, which changes the last bit of about one distance in ten.  So
// the running sum is never written as an add of a product: it is
//     acc = fma.rn(one, sq, acc)
// where `one` is 1.0 passed in as a kernel argument.  1 * sq is exact, so
// this is exactly one rounding of acc + sq (the add), and because `one` is
// unknown when the kernel is compiled the optimiser can neither turn it back
// into an add nor fold the multiply that produced sq into it.  The subtract
// and the square are plain round-to-nearest packed operations; packed forms
// round each lane exactly like the scalar instruction, so one lane of a
// packed distance is bit-identical to the scalar distance below.

__device__ __forceinline__ float add_rn(float a, float b)
{
    float r;
    asm("add.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float mul_rn(float a, float b)
{
    float r;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float fma_rn(float a, float b, float c)
{
    float r;
    asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float2 add2_rn(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "add.rn.f32x2 pd, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %5};\n\t"
        "mov.b64 pc, {%6, %7};\n\t"
        "fma.rn.f32x2 pd, pa, pb, pc;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// Squared distances of one centroid (negated, duplicated: nc[i] = (-c_i, -c_i))
// to the two sub-vectors packed in xp[i] = (x_i, x'_i).  Ascending i; the
// subtract, the square and the sum each round to nearest on their own.
// `one` must hold (1.0f, 1.0f) (see above).
template <int SUB>
__device__ __forceinline__ float2 pair_dist(const float2 (&xp)[SUB], const float2 (&nc)[SUB],
                                            float2 one)
{
    float2 d = add2_rn(xp[0], nc[0]);
    float2 acc = mul2_rn(d, d);
#pragma unroll
    for (int i = 1; i < SUB; ++i) {
        d = add2_rn(xp[i], nc[i]);
        acc = fma2_rn(one, mul2_rn(d, d), acc);
    }
    return acc;
}

// The same distance for one sub-vector, scalar.  Bit-identical to one lane
// of pair_dist.  `one` must be 1.0f.
template <int SUB>
__device__ __forceinline__ float one_dist(const float (&x)[SUB], const float (&nc)[SUB], float one)
{
    float d = add_rn(x[0], nc[0]);
    float acc = mul_rn(d, d);
#pragma unroll
    for (int i = 1; i < SUB; ++i) {
        d = add_rn(x[i], nc[i]);
        acc = fma_rn(one, mul_rn(d, d), acc);
    }
    return acc;
}

// ------------------------------------------------------------------ codebook staging

// Shared-memory codebook layout: centroids in groups of GC; centroid c of
// group g occupies SUB/2 float4 = {-c_i, -c_i, -c_{i+1}, -c_{i+1}}; each group
// is followed by one padding float4 so that groups start on different banks
// (the deferred strategy's re-evaluation reads one group per lane).
template <int SUB, int GC>
struct CbLayout {
    static constexpr int kF4PerCentroid = SUB / 2;
    static constexpr int kGroupStride = GC * kF4PerCentroid + 1;  // float4 units
    __host__ __device__ static int groups(int n_centroids) { return (n_centroids + GC - 1) / GC; }
    __host__ __device__ static size_t bytes(int n_centroids)
    {
        return (size_t)groups(n_centroids) * kGroupStride * sizeof(float4);
    }
};

// Stage codebook cb[n_centroids][SUB] (global, type T) into shared memory.
// Rows past n_centroids (padding up to a multiple of GC) are NaN: their
// distance is NaN and never wins.
template <typename T, int SUB, int GC>
__device__ __forceinline__ void stage_codebook(const T *__restrict__ cb, int n_centroids,
                                               float4 *__restrict__ s)
{
    using L = CbLayout<SUB, GC>;
    const int n_pad = L::groups(n_centroids) * GC;
    const int total = n_pad * (SUB / 2);
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
        const int c = e / (SUB / 2);
        const int k = e - c * (SUB / 2);
        float a = __int_as_float(0x7fc00000), b = a;
        if (c < n_centroids) {
            a = -widen(cb[(size_t)c * SUB + 2 * k]);
            b = -widen(cb[(size_t)c * SUB + 2 * k + 1]);
        }
        s[(c / GC) * L::kGroupStride + (c % GC) * L::kF4PerCentroid + k] = make_float4(a, a, b, b);
    }
}

template <int SUB>
__device__ __forceinline__ void read_centroid(const float4 *__restrict__ p, float2 (&nc)[SUB])
{
#pragma unroll
    for (int k = 0; k < SUB / 2; ++k) {
        const float4 q = p[k];
        nc[2 * k] = make_float2(q.x, q.y);
        nc[2 * k + 1] = make_float2(q.z, q.w);
    }
}

template <int SUB>
__device__ __forceinline__ void read_centroid_scalar(const float4 *__restrict__ p,
                                                     float (&nc)[SUB])
{
#pragma unroll
    for (int k = 0; k < SUB / 2; ++k) {
        const float4 q = p[k];
        nc[2 * k] = q.x;
        nc[2 * k + 1] = q.z;
    }
}

// ------------------------------------------------------------------ fast kernel

// Launch: grid.x = n_groups * tiles_per_group, block = THREADS; dynamic shared
// memory = CbLayout<SUB, GC>::bytes(n_centroids); `one` = 1.0f.  Block b encodes tile
// (b % tiles_per_group) of group (b / tiles_per_group); a tile is THREADS * R
// consecutive rows of that group.  Requires x aligned to SUB * sizeof(T)
// bytes (16 bytes at most), 1 <= n_centroids and the shared memory to fit.
template <typename T, int SUB, int R, int THREADS, int MODE, int GC, typename OutT = uint32_t>
__global__ void __launch_bounds__(THREADS)
    encode_fast(const T *__restrict__ x, const T *__restrict__ codebooks, int64_t n_per_group,
                int32_t n_centroids, int64_t tiles_per_group, float one,
                OutT *__restrict__ out)
{
    static_assert(R % 2 == 0, "rows per thread come in packed pairs");
    static_assert(SUB % 2 == 0, "sub_dim must be even for the packed layout");
    static_assert(GC % 2 == 0, "centroid groups come in pairs");
    using L = CbLayout<SUB, GC>;
    extern __shared__ float4 smem[];

    const int64_t g = blockIdx.x / tiles_per_group;
    const int64_t tile = blockIdx.x - g * tiles_per_group;
    const T *__restrict__ cb = codebooks + (size_t)g * (size_t)n_centroids * SUB;
    const T *__restrict__ xg = x + (size_t)g * (size_t)n_per_group * SUB;
    OutT *__restrict__ og = out + (size_t)g * (size_t)n_per_group;
    const int64_t row0 = tile * (int64_t)(THREADS * R) + threadIdx.x;

    // Rows of this thread: row0 + r * THREADS.  Rows past the end compute on
    // zeros and are not stored.
    float2 xp[R / 2][SUB];
#pragma unroll
    for (int rp = 0; rp < R / 2; ++rp) {
        float a[SUB], b[SUB];
        const int64_t ra = row0 + (int64_t)(2 * rp) * THREADS;
        const int64_t rb = ra + THREADS;
        if (ra < n_per_group) {
            load_row<T, SUB>(xg + (size_t)ra * SUB, a);
        } else {
#pragma unroll
            for (int i = 0; i < SUB; ++i) a[i] = 0.f;
        }
        if (rb < n_per_group) {
            load_row<T, SUB>(xg + (size_t)rb * SUB, b);
        } else {
#pragma unroll
            for (int i = 0; i < SUB; ++i) b[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < SUB; ++i) xp[rp][i] = make_float2(a[i], b[i]);
    }

    stage_codebook<T, SUB, GC>(cb, n_centroids, smem);
    __syncthreads();

    const int n_cgroups = L::groups(n_centroids);
    const float2 one2 = make_float2(one, one);
    uint32_t result[R];

    if constexpr (MODE == kDirect) {
        float best[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            best[r] = __int_as_float(0x7f800000);
            result[r] = 0;
        }
        for (int cg = 0; cg < n_cgroups; ++cg) {
            const float4 *gp = smem + cg * L::kGroupStride;
#pragma unroll
            for (int cc = 0; cc < GC; ++cc) {
                float2 nc[SUB];
                read_centroid<SUB>(gp + cc * L::kF4PerCentroid, nc);
                const uint32_t cid = (uint32_t)(cg * GC + cc);
#pragma unroll
                for (int rp = 0; rp < R / 2; ++rp) {
                    const float2 dd = pair_dist<SUB>(xp[rp], nc, one2);
                    if (dd.x < best[2 * rp]) {
                        best[2 * rp] = dd.x;
                        result[2 * rp] = cid;
                    }
                    if (dd.y < best[2 * rp + 1]) {
                        best[2 * rp + 1] = dd.y;
                        result[2 * rp + 1] = cid;
                    }
                }
            }
        }
    } else {
        float run[R], prev[R];
        int win[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            run[r] = __int_as_float(0x7f800000);
            prev[r] = run[r];
            win[r] = 0;
        }
        for (int cg = 0; cg < n_cgroups; ++cg) {
            const float4 *gp = smem + cg * L::kGroupStride;
#pragma unroll
            for (int cc = 0; cc < GC; cc += 2) {
                float2 na[SUB], nb[SUB];
                read_centroid<SUB>(gp + cc * L::kF4PerCentroid, na);
                read_centroid<SUB>(gp + (cc + 1) * L::kF4PerCentroid, nb);
#pragma unroll
                for (int rp = 0; rp < R / 2; ++rp) {
                    const float2 da = pair_dist<SUB>(xp[rp], na, one2);
                    const float2 db = pair_dist<SUB>(xp[rp], nb, one2);
                    run[2 * rp] = min3(run[2 * rp], da.x, db.x);
                    run[2 * rp + 1] = min3(run[2 * rp + 1], da.y, db.y);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                win[r] = run[r] < prev[r] ? cg : win[r];
                prev[r] = run[r];
            }
        }
        // Re-evaluate the winning group of each row, highest index first, so
        // the last match kept is the lowest index with the minimal distance.
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float xr[SUB];
#pragma unroll
            for (int i = 0; i < SUB; ++i) xr[i] = (r & 1) ? xp[r / 2][i].y : xp[r / 2][i].x;
            uint32_t id = 0;
            if (run[r] < __int_as_float(0x7f800000)) {
                const float4 *gp = smem + win[r] * L::kGroupStride;
#pragma unroll 2
                for (int cc = GC - 1; cc >= 0; --cc) {
                    float nc[SUB];
                    read_centroid_scalar<SUB>(gp + cc * L::kF4PerCentroid, nc);
                    if (one_dist<SUB>(xr, nc, one) == run[r]) id = (uint32_t)(win[r] * GC + cc);
                }
            }
            result[r] = id;
        }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + (int64_t)r * THREADS;
        if (row < n_per_group) store_index(og + row, result[r]);
    }
}

// ------------------------------------------------------------------ general kernel

// Any sub_dim, any n_centroids, x and codebooks aligned to their element
// size only: one thread per row, scalar fp32 arithmetic, x and the codebook
// read through the read-only cache.
// Launch: grid.x = ceil(n_groups * n_per_group / blockDim.x); `one` = 1.0f.
template <typename T, typename OutT = uint32_t>
__global__ void encode_general(const T *__restrict__ x, const T *__restrict__ codebooks,
                               int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                               int32_t sub_dim, float one, OutT *__restrict__ out)
{
    const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= n_groups * n_per_group) return;
    const int64_t g = row / n_per_group;
    const T *__restrict__ cb = codebooks + (size_t)g * (size_t)n_centroids * sub_dim;
    const T *__restrict__ xr = x + (size_t)row * sub_dim;
    float best = __int_as_float(0x7f800000);
    uint32_t idx = 0;
    for (int32_t c = 0; c < n_centroids; ++c) {
        const T *__restrict__ cr = cb + (size_t)c * sub_dim;
        float d = add_rn(widen(__ldg(xr)), -widen(__ldg(cr)));
        float acc = mul_rn(d, d);
        for (int32_t i = 1; i < sub_dim; ++i) {
            d = add_rn(widen(__ldg(xr + i)), -widen(__ldg(cr + i)));
            acc = fma_rn(one, mul_rn(d, d), acc);
        }
        if (acc < best) {
            best = acc;
            idx = (uint32_t)c;
        }
    }
    store_index(out + row, idx);
}

}  // namespace vqk
