// vq_filter.cuh -- exact product-VQ encode with less arithmetic: screen every
// centroid with a fused multiply-add score, bound the screening error
// rigorously, and evaluate the exact fp32 distance formula only where the
// bound cannot rule a centroid out.  The indices are those of the exact
// definition ("I Wrote a Metal Kernel to Stop My Mac From OOMing", section
// "The Kernel: 18 Lines of MSL"), bit for bit.
//
// Why it is exact.  For a row x and centroid c, D(c) = |x - c|^2 =
// |x|^2 + S(c) with S(c) = |c|^2 - 2 x.c, so the centroids order by S.
//   1. Screening: s~(c) = fma(x_SUB-1, w_SUB-1, ... fma(x_0, w_0, n~(c))), with
//      w_i = -2 c_i (exact) and n~(c) the fp32 |c|^2 (one multiply, SUB-1
//      fmas).  Each fma rounds once, so |s~(c) - S(c)| <= (2 + g) g (|c|^2 +
//      sum_i |x_i| |c_i|) with g = gamma_SUB, gamma_k = k u / (1 - k u),
//      u = 2^-24.  With C2 = max_c n~(c) and A_i = max_c |c_i| this is at
//      most B(x) = 4 gamma_SUB (C2 + sum_i |x_i| A_i) for every c.
//   2. The exact fp32 distance D32(c) lies within a factor (1 +- e) of D(c),
//      e = gamma_{SUB+2} (SUB+2 roundings on each nonnegative term).
//   3. Let m = argmin s~ and c* the oracle's centroid.  D32(c*) <= D32(m)
//      gives S(c*) <= S(m) + 2 e/(1-e) D(m), hence s~(c*) <= s~(m) + 2 B +
//      2 e/(1-e) D(m), and D(m) <= |x|^2 + s~(m) + B.  The kernel uses
//      thr = s~(m) + 2 B + 4 e Dmax + 2^-100 with Dmax = |x|^2 + s~(m) + B;
//      the factor 2 of slack absorbs the rounding of computing B, Dmax and
//      thr themselves, and 2^-100 covers gradual underflow.  So every group
//      holding c* has its least s~ at or below thr.
//   4. Per row the kernel keeps the least s~ of each group of GC centroids
//      and the three smallest group minima m1 <= m2 <= m3.  If m2 > thr only
//      group g1 can hold c*; if m3 > thr only g1 or g2.  It evaluates the
//      exact formula on those GC (or 2 GC) centroids in ascending index order
//      with a strict "<": the lexicographic (D32, index) minimum over a set
//      that contains c* is c*.
//   5. Rows with three or more candidate groups, or whose bound is not finite
//      or is near fp32 overflow (NaN / inf inputs, huge values), are queued in
//      shared memory; at the end of the block whole warps scan them exactly
//      (32 lanes split the centroids, then a shuffle reduction of
//      (distance, index), lowest index winning ties).  No global scratch.
#pragma once

#include "vq_check.cuh"
#include "vq_kernels.cuh"

namespace vqk {

template <int SUB, int GC>
struct FilterLayout {
    // Shared memory, in float4 units:
    //   screening weights: per centroid SUB/2 float4 {w_i, w_i, w_i+1, w_i+1}
    //   screening norms:   per centroid pair {n_c, n_c, n_c+1, n_c+1}
    //   exact values:      per group GC * SUB/4 float4 of -c_i, then 1 pad float4
    // then SUB + 1 uint32 maxima (C2, A_0..A_SUB-1), a queue counter and the
    // queue (one uint32 per row of the tile).
    static constexpr int kW4 = SUB / 2;
    static constexpr int kX4 = SUB / 4;
    static constexpr int kGroupStride = GC * kX4 + 1;
    __host__ __device__ static int groups(int nc) { return (nc + GC - 1) / GC; }
    __host__ __device__ static int padded(int nc) { return groups(nc) * GC; }
    __host__ __device__ static size_t n_off(int nc) { return (size_t)padded(nc) * kW4; }
    __host__ __device__ static size_t x_off(int nc) { return n_off(nc) + padded(nc) / 2; }
    __host__ __device__ static size_t f4_total(int nc)
    {
        return x_off(nc) + (size_t)groups(nc) * kGroupStride;
    }
    __host__ __device__ static size_t bytes(int nc, int tile_rows)
    {
        return f4_total(nc) * sizeof(float4) + (SUB + 2) * sizeof(uint32_t) +
               (size_t)tile_rows * sizeof(uint32_t);
    }
};

// gamma_k = k u / (1 - k u), u = 2^-24
__device__ __forceinline__ float gamma_u(int k)
{
    return k * 5.9604645e-8f / (1.0f - k * 5.9604645e-8f);
}

// Row `row` of group g divided element-wise by its channels' smooth factors
// (SMOOTH only): channels (row % smooth_ns) * SUB + i of smooth[g][.], fp32
// division rounded to nearest.
template <int SUB, bool SMOOTH>
__device__ __forceinline__ void smooth_row(float (&v)[SUB], const float *__restrict__ sg,
                                           int64_t row, int32_t smooth_ns)
{
    if constexpr (SMOOTH) {
        const float *f = sg + (size_t)(row % smooth_ns) * SUB;
#pragma unroll
        for (int i = 0; i < SUB; ++i) v[i] = __fdiv_rn(v[i], __ldg(f + i));
    }
}

// Launch: grid.x = n_groups * tiles_per_group, block = THREADS, dynamic shared
// memory = FilterLayout<SUB, GC>::bytes(n_centroids, THREADS * R); `one` =
// 1.0f.  Same tiling and alignment requirements as encode_fast.  With SMOOTH,
// every row is first divided by its per-channel smooth factors (`smooth`
// [n_groups][smooth_ns * SUB]; groups are whole key vectors of smooth_ns
// rows); the bound below then holds for the divided row, which is what is
// encoded.  Without SMOOTH, `smooth` and `smooth_ns` are unused.
template <typename T, int SUB, int R, int THREADS, int GC, typename OutT = uint32_t,
          bool SMOOTH = false>
__global__ void __launch_bounds__(THREADS)
    encode_filter(const T *__restrict__ x, const T *__restrict__ codebooks, int64_t n_per_group,
                  int32_t n_centroids, int64_t tiles_per_group, float one,
                  OutT *__restrict__ out, const float *__restrict__ smooth, int32_t smooth_ns)
{
    static_assert(R % 2 == 0 && SUB % 4 == 0 && GC % 2 == 0, "layout constraints");
    using L = FilterLayout<SUB, GC>;
    constexpr int kTile = THREADS * R;
    constexpr uint32_t kQueued = 0xffffffffu;
    extern __shared__ float4 smem[];
    const int n_pad = L::padded(n_centroids);
    const int n_cg = L::groups(n_centroids);
    float4 *sw = smem;
    float4 *sn = smem + L::n_off(n_centroids);
    float4 *sx = smem + L::x_off(n_centroids);
    uint32_t *smax = reinterpret_cast<uint32_t *>(smem + L::f4_total(n_centroids));
    uint32_t *qcount = smax + SUB + 1;
    uint32_t *queue = qcount + 1;

    const int64_t g = blockIdx.x / tiles_per_group;
    const int64_t tile = blockIdx.x - g * tiles_per_group;
    const T *__restrict__ cb = codebooks + (size_t)g * (size_t)n_centroids * SUB;
    const T *__restrict__ xg = x + (size_t)g * (size_t)n_per_group * SUB;
    OutT *__restrict__ og = out + (size_t)g * (size_t)n_per_group;
    const float *__restrict__ sg = SMOOTH ? smooth + (size_t)g * (size_t)smooth_ns * SUB : nullptr;
    const int64_t row0 = tile * (int64_t)kTile + threadIdx.x;

    // buffer extents, for the checked build's bounds checks (vq_check.cuh)
    const int64_t n_groups_all = gridDim.x / tiles_per_group;
    const int64_t nx = n_groups_all * n_per_group * SUB, nout = n_groups_all * n_per_group;
    const uint64_t f4_total = L::f4_total(n_centroids);
    constexpr uint32_t kRowAlign = SUB * sizeof(T) < 16 ? SUB * sizeof(T) : 16;  // load_row
    if constexpr (kChecked) {
        // the layout inside the launch's shared memory, the block inside the
        // grid, its smooth factors inside theirs: else the block does nothing
        if (!dyn_smem_ok(smem, L::bytes(n_centroids, kTile), 16) || !index_ok(g, n_groups_all) ||
            (SMOOTH && !VQ_SPAN(sg, (int64_t)smooth_ns * SUB, smooth, n_groups_all * smooth_ns * SUB)))
            return;  // block-uniform
    }

    // Rows of this thread: row0 + r * THREADS, rows 2rp and 2rp+1 packed in
    // one float2.  Rows past the end compute on zeros and are not stored.
    float2 xp[R / 2][SUB];
#pragma unroll
    for (int rp = 0; rp < R / 2; ++rp) {
        float a[SUB], b[SUB];
        const int64_t ra = row0 + (int64_t)(2 * rp) * THREADS;
        const int64_t rb = ra + THREADS;
        if (ra < n_per_group && VQ_VSPAN(xg + (size_t)ra * SUB, SUB, x, nx, kRowAlign)) {
            load_row<T, SUB>(xg + (size_t)ra * SUB, a);
            smooth_row<SUB, SMOOTH>(a, sg, ra, smooth_ns);
        } else {
#pragma unroll
            for (int i = 0; i < SUB; ++i) a[i] = 0.f;
        }
        if (rb < n_per_group && VQ_VSPAN(xg + (size_t)rb * SUB, SUB, x, nx, kRowAlign)) {
            load_row<T, SUB>(xg + (size_t)rb * SUB, b);
            smooth_row<SUB, SMOOTH>(b, sg, rb, smooth_ns);
        } else {
#pragma unroll
            for (int i = 0; i < SUB; ++i) b[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < SUB; ++i) xp[rp][i] = make_float2(a[i], b[i]);
    }

    // ---- stage the codebook (both layouts) and its maxima
    if (threadIdx.x < SUB + 2) smax[threadIdx.x] = 0u;  // maxima and queue counter
    __syncthreads();
    for (int c = threadIdx.x; c < n_pad; c += THREADS) {
        const bool real = c < n_centroids;
        const bool cb_ok = !real || VQ_SPAN(cb + (size_t)c * SUB, SUB, codebooks, n_groups_all * n_centroids * SUB);
        float v[SUB];
#pragma unroll
        for (int i = 0; i < SUB; ++i)
            v[i] = real && cb_ok ? widen(cb[(size_t)c * SUB + i]) : __int_as_float(0x7fc00000);
        float nrm = mul_rn(v[0], v[0]);
#pragma unroll
        for (int i = 1; i < SUB; ++i) nrm = fma_rn(v[i], v[i], nrm);
#pragma unroll
        for (int k = 0; k < SUB / 2; ++k) {
            const float w0 = -2.0f * v[2 * k], w1 = -2.0f * v[2 * k + 1];
            if (VQ_SPAN(sw + (size_t)c * L::kW4 + k, 1, sw, L::n_off(n_centroids)))
                sw[(size_t)c * L::kW4 + k] = make_float4(w0, w0, w1, w1);
        }
        if (span_ok(reinterpret_cast<float2 *>(sn) + c, 8, sn, (L::x_off(n_centroids) - L::n_off(n_centroids)) * 16, 8))
            reinterpret_cast<float2 *>(sn)[c] = make_float2(nrm, nrm);
        float4 *ex = sx + (c / GC) * L::kGroupStride + (c % GC) * L::kX4;
#pragma unroll
        for (int k = 0; k < SUB / 4; ++k)
            if (VQ_SPAN(ex + k, 1, sx, f4_total - L::x_off(n_centroids)))
                ex[k] = make_float4(-v[4 * k], -v[4 * k + 1], -v[4 * k + 2], -v[4 * k + 3]);
        if (real) {
            // nonnegative floats (and NaN, which sorts above +inf) order as
            // their bit patterns
            atomicMax(&smax[0], __float_as_uint(nrm));
#pragma unroll
            for (int i = 0; i < SUB; ++i) atomicMax(&smax[1 + i], __float_as_uint(fabsf(v[i])));
        }
    }
    __syncthreads();

    // ---- screening: the three smallest group minima of s~ per row
    const float kInf = __int_as_float(0x7f800000);
    float m1[R], m2[R], m3[R];
    int g1[R], g2[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        m1[r] = m2[r] = m3[r] = kInf;
        g1[r] = g2[r] = 0;
    }
    for (int cg = 0; cg < n_cg; ++cg) {
        float run[R];
#pragma unroll
        for (int r = 0; r < R; ++r) run[r] = kInf;
#pragma unroll
        for (int cc = 0; cc < GC; cc += 2) {
            const int c = cg * GC + cc;
            const float4 nn = VQ_SPAN(sn + c / 2, 1, sn, L::x_off(n_centroids) - L::n_off(n_centroids))
                                  ? sn[c / 2] : make_float4(0.f, 0.f, 0.f, 0.f);
            float2 wa[SUB], wb[SUB];
#pragma unroll
            for (int k = 0; k < SUB / 2; ++k) {
                const bool w_ok = VQ_SPAN(sw + (size_t)c * L::kW4 + k, L::kW4 + 1, sw, L::n_off(n_centroids));
                const float4 qa = w_ok ? sw[(size_t)c * L::kW4 + k] : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 qb = w_ok ? sw[(size_t)(c + 1) * L::kW4 + k] : make_float4(0.f, 0.f, 0.f, 0.f);
                wa[2 * k] = make_float2(qa.x, qa.y);
                wa[2 * k + 1] = make_float2(qa.z, qa.w);
                wb[2 * k] = make_float2(qb.x, qb.y);
                wb[2 * k + 1] = make_float2(qb.z, qb.w);
            }
#pragma unroll
            for (int rp = 0; rp < R / 2; ++rp) {
                float2 sa = make_float2(nn.x, nn.y);
                float2 sb = make_float2(nn.z, nn.w);
#pragma unroll
                for (int i = 0; i < SUB; ++i) {
                    sa = fma2_rn(xp[rp][i], wa[i], sa);
                    sb = fma2_rn(xp[rp][i], wb[i], sb);
                }
                run[2 * rp] = min3(run[2 * rp], sa.x, sb.x);
                run[2 * rp + 1] = min3(run[2 * rp + 1], sa.y, sb.y);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float gm = run[r];
            const bool p1 = gm < m1[r];
            const bool p2 = gm < m2[r];
            m3[r] = p2 ? m2[r] : fminf(m3[r], gm);
            m2[r] = p1 ? m1[r] : (p2 ? gm : m2[r]);
            g2[r] = p1 ? g1[r] : (p2 ? cg : g2[r]);
            m1[r] = p1 ? gm : m1[r];
            g1[r] = p1 ? cg : g1[r];
        }
    }

    // ---- bound, candidate groups, exact re-evaluation
    const float c2 = __uint_as_float(smax[0]);
    float amax[SUB];
#pragma unroll
    for (int i = 0; i < SUB; ++i) amax[i] = __uint_as_float(smax[1 + i]);
    const float kB = 4.0f * gamma_u(SUB);
    const float kD = 4.0f * gamma_u(SUB + 2);
    const float kTiny = 7.8886091e-31f;  // 2^-100
    uint32_t result[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float xr[SUB];
#pragma unroll
        for (int i = 0; i < SUB; ++i) xr[i] = (r & 1) ? xp[r / 2][i].y : xp[r / 2][i].x;
        float sabs = 0.f, xx = 0.f;
#pragma unroll
        for (int i = 0; i < SUB; ++i) {
            sabs = fmaf(fabsf(xr[i]), amax[i], sabs);
            xx = fmaf(xr[i], xr[i], xx);
        }
        const float base = c2 + sabs;
        const float bnd = kB * base + kTiny;
        const float dmax = fmaxf(0.f, xx + m1[r] + bnd);
        const float thr = m1[r] + (2.0f * bnd + kD * dmax + kTiny);
        // false for NaN or inf anywhere in the row or the codebook, and for
        // magnitudes where an fp32 distance could overflow
        const bool ok = base < 1e30f && dmax < 1e37f;
        const bool two = m2[r] <= thr;
        const int64_t row = row0 + (int64_t)r * THREADS;
        uint32_t id = 0;
        if (!ok || m3[r] <= thr) {
            id = kQueued;
            if (row < n_per_group) {
                const uint32_t k = atomicAdd(qcount, 1u);
                if (VQ_SPAN(queue + k, 1, queue, kTile)) queue[k] = (uint32_t)(r * THREADS + threadIdx.x);
            }
        } else {
            const int ga = two ? min(g1[r], g2[r]) : g1[r];
            const int gb = two ? max(g1[r], g2[r]) : -1;
            float best = kInf;
            for (int pass = 0; pass < 2; ++pass) {
                const int gsel = pass == 0 ? ga : gb;
                if (gsel < 0) break;
                const float4 *gp = sx + gsel * L::kGroupStride;
#pragma unroll 4
                for (int cc = 0; cc < GC; ++cc) {
                    float nc[SUB];
#pragma unroll
                    for (int k = 0; k < SUB / 4; ++k) {
                        const float4 q = VQ_SPAN(gp + cc * L::kX4 + k, 1, sx, f4_total - L::x_off(n_centroids))
                                             ? gp[cc * L::kX4 + k] : make_float4(0.f, 0.f, 0.f, 0.f);
                        nc[4 * k] = q.x;
                        nc[4 * k + 1] = q.y;
                        nc[4 * k + 2] = q.z;
                        nc[4 * k + 3] = q.w;
                    }
                    const float d = one_dist<SUB>(xr, nc, one);
                    if (d < best) {
                        best = d;
                        id = (uint32_t)(gsel * GC + cc);
                    }
                }
            }
        }
        result[r] = id;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + (int64_t)r * THREADS;
        if (row < n_per_group && result[r] != kQueued && VQ_SPAN(og + row, 1, out, nout))
            store_index(og + row, result[r]);
    }

    // ---- queued rows: one warp per row, exact scan over all centroids
    __syncthreads();
    const uint32_t nq = *qcount;
    const int lane = threadIdx.x & 31;
    for (uint32_t q = threadIdx.x >> 5; q < nq; q += THREADS / 32) {
        if (!VQ_SPAN(queue + q, 1, queue, kTile)) break;  // warp-uniform
        const int64_t row = tile * (int64_t)kTile + queue[q];
        if (!VQ_SPAN(xg + (size_t)row * SUB, SUB, x, nx)) continue;  // warp-uniform
        float xr[SUB];
#pragma unroll
        for (int i = 0; i < SUB; ++i) xr[i] = widen(xg[(size_t)row * SUB + i]);
        smooth_row<SUB, SMOOTH>(xr, sg, row, smooth_ns);
        float best = kInf;
        uint32_t id = kQueued;
        for (int c = lane; c < n_centroids; c += 32) {
            const float4 *cp = sx + (c / GC) * L::kGroupStride + (c % GC) * L::kX4;
            float nc[SUB];
#pragma unroll
            for (int k = 0; k < SUB / 4; ++k) {
                const float4 qv = VQ_SPAN(cp + k, 1, sx, f4_total - L::x_off(n_centroids))
                                      ? cp[k] : make_float4(0.f, 0.f, 0.f, 0.f);
                nc[4 * k] = qv.x;
                nc[4 * k + 1] = qv.y;
                nc[4 * k + 2] = qv.z;
                nc[4 * k + 3] = qv.w;
            }
            const float d = one_dist<SUB>(xr, nc, one);
            if (d < best) {
                best = d;
                id = (uint32_t)c;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, off);
            const uint32_t oi = __shfl_xor_sync(0xffffffffu, id, off);
            if (ob < best || (ob == best && oi < id)) {
                best = ob;
                id = oi;
            }
        }
        // no finite, non-NaN distance anywhere: index 0, as the definition gives
        if (lane == 0 && VQ_SPAN(og + row, 1, out, nout)) store_index(og + row, id == kQueued ? 0u : id);
    }
}

}  // namespace vqk
