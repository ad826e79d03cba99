// vq_attn.cuh -- decode attention straight from product-VQ codes ("I Wrote a
// Metal Kernel to Stop My Mac From OOMing", section "What's Next: Phase 2":
// a per-query lookup table of q against the codebook, scores read from it by
// the key codes without rebuilding the keys, and the softmax-weighted value
// sum in the same pass; "Metal 4 TensorOps ...", section "The Kernel's Hot
// Path", spells the table out as one dot product per (sub-space, centroid)).
//
// For one query q (head dim D = NS * SUB) against a cache of T tokens stored
// as 8-bit codes, with kappa = scale * log2(e):
//   LUT[s][c]    = kappa * sum_i q[s*SUB + i] * Kcb[c][i]        (fp32)
//   score[t]     = sum_s LUT[s][kcode[t][s]]          = kappa * q . K^[t]
//   p[t]         = 2^(score[t] - max) / sum_t' 2^(score[t'] - max)
//   out[s*SUB+i] = sum_t p[t] * Vcb[vcode[t][s]][i]    = sum_t p[t] V^[t]
// (2^(kappa x) = e^(scale x), so this is the usual softmax.)  The value sum is
// regrouped by code: W[s][c] = sum of 2^(score - max) over the tokens whose
// value code in sub-space s is c, so a token costs NS shared-memory adds
// instead of D multiply-adds, and out = (W @ Vcb) / l at the end.
//
// GB300 shape: a block owns GPB query heads of one KV head (grouped-query
// attention: they share that head's codes and codebooks) and one run of
// CHUNK-token chunks, so each code row is read from HBM once for all of them.
// Tables and W sit in shared memory with a row stride of kLutStride floats:
// entries past n_centroids stay zero, so a code >= n_centroids reads a zero
// key row and adds to a value row that is never read (the decode of such a
// code is a zero row).  Scores of a chunk stay in registers between the max
// and the accumulation; W is rescaled when a later chunk raises the running
// maximum (online softmax at chunk granularity).  Each block writes a partial
// (max, sum, out[D]) per query head to the caller's workspace; attn_combine
// merges the partials (flash-decoding).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace vqk {

constexpr int kLutStride = 260;  // >= 256 codes; 4 * s spreads sub-spaces over banks
constexpr int kAttnMaxHeads = 8;
constexpr int kAttnTokPerThread = 4;

struct AttnShape {
    int64_t batch;
    int32_t heads_q, heads_kv, head_dim, sub_dim, n_centroids;
    int64_t tokens;           // cached tokens T
    int64_t first_token;      // first attended token (sliding window), else 0
    int64_t chunks;           // ceil((T - first_token) / CHUNK)
    int32_t heads_per_block;  // GPB
    int32_t splits;           // chunk runs per (batch, KV head, head group)
    float kappa;              // scale * log2(e)
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f32(float &d, float v) { d = v; }
__device__ __forceinline__ void from_f32(__half &d, float v) { d = __float2half_rn(v); }
__device__ __forceinline__ void from_f32(__nv_bfloat16 &d, float v) { d = __float2bfloat16_rn(v); }

// Shared memory: LUT [GPB][NS][kLutStride], W [GPB][NS][kLutStride], block
// reduction scratch [3][GPB][32] (two alternating max buffers, one sum).
__host__ __device__ inline size_t attn_smem_bytes(int gpb, int ns)
{
    return ((size_t)2 * gpb * ns * kLutStride + 3 * (size_t)gpb * 32) * sizeof(float);
}

// Code row of one token as 32-bit words (NS bytes, NS % 4 == 0, row address
// aligned to the largest power of two dividing NS, at most 16).
template <int NS>
__device__ __forceinline__ void load_code_row(const uint8_t *p, uint32_t (&w)[NS / 4])
{
    if constexpr (NS % 16 == 0) {
#pragma unroll
        for (int k = 0; k < NS / 16; ++k) {
            const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p) + k);
            w[4 * k] = v.x, w[4 * k + 1] = v.y, w[4 * k + 2] = v.z, w[4 * k + 3] = v.w;
        }
    } else if constexpr (NS % 8 == 0) {
#pragma unroll
        for (int k = 0; k < NS / 8; ++k) {
            const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(p) + k);
            w[2 * k] = v.x, w[2 * k + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < NS / 4; ++k) w[k] = __ldcs(reinterpret_cast<const uint32_t *>(p) + k);
    }
}

__device__ __forceinline__ uint32_t code_at(uint32_t w, int k) { return (w >> (8 * k)) & 0xffu; }

// Launch: grid.x = batch * heads_kv * (heads_q / heads_kv / GPB) * splits,
// block = THREADS, dynamic shared memory attn_smem_bytes(GPB, NS).  NS (the
// number of sub-spaces, head_dim / sub_dim) is a compile-time multiple of 4;
// code rows are NS bytes apart and the code arrays are 16-byte aligned.
// Partial of (b, hq, split) at part[((b * heads_q + hq) * splits + split) *
// (D + 2)]: {0: max (log2 domain), 1: sum, 2..: unnormalised out}.
template <typename T, int THREADS, int NS>
__global__ void __launch_bounds__(THREADS)
    attn_partial(const T *__restrict__ q, const uint8_t *__restrict__ kcodes,
                 const T *__restrict__ kcb, const uint8_t *__restrict__ vcodes,
                 const T *__restrict__ vcb, AttnShape sh, float *__restrict__ part)
{
    constexpr int TPT = kAttnTokPerThread;
    constexpr int CHUNK = THREADS * TPT;
    constexpr int G = kAttnMaxHeads;
    constexpr int NW = THREADS / 32;
    constexpr float kNegInf = -__builtin_huge_valf();
    extern __shared__ float smem_attn[];
    const int sub = sh.sub_dim;
    const int nc = sh.n_centroids;
    const int gpb = sh.heads_per_block;
    const int qpk = sh.heads_q / sh.heads_kv;  // query heads per KV head
    const int hgroups = qpk / gpb;
    const int tab = NS * kLutStride;           // floats per head
    float *lut = smem_attn;                    // [gpb][NS][kLutStride]
    float *wsum = lut + (size_t)gpb * tab;     // [gpb][NS][kLutStride]
    float *red = wsum + (size_t)gpb * tab;     // [3][gpb][32]

    int64_t bid = blockIdx.x;
    const int split = (int)(bid % sh.splits);
    bid /= sh.splits;
    const int hg = (int)(bid % hgroups);
    bid /= hgroups;
    const int hkv = (int)(bid % sh.heads_kv);
    const int64_t b = bid / sh.heads_kv;
    const int hq0 = hkv * qpk + hg * gpb;

    const T *kc = kcb + (size_t)hkv * nc * sub;
    const T *vc = vcb + (size_t)hkv * nc * sub;
    const size_t cache_off = ((size_t)b * sh.heads_kv + hkv) * (size_t)sh.tokens * NS;
    const uint8_t *kb = kcodes + cache_off;
    const uint8_t *vb = vcodes + cache_off;

    // chunks [c0, c1) of the attended span belong to this block
    const int64_t c0 = sh.chunks * split / sh.splits;
    const int64_t c1 = sh.chunks * (split + 1) / sh.splits;

    // ---- tables (kappa folded in; zero past n_centroids) and zeroed W
    for (int e = threadIdx.x; e < gpb * tab; e += THREADS) {
        const int c = e % kLutStride;
        const int s = (e / kLutStride) % NS;
        const int g = e / tab;
        float acc = 0.f;
        if (c < nc) {
            const T *qv = q + ((size_t)b * sh.heads_q + hq0 + g) * sh.head_dim + (size_t)s * sub;
            const T *cv = kc + (size_t)c * sub;
            for (int i = 0; i < sub; ++i) acc = fmaf(to_f32(qv[i]), to_f32(cv[i]), acc);
        }
        lut[e] = acc * sh.kappa;
        wsum[e] = 0.f;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float m_run[G], l_run[G];
#pragma unroll
    for (int g = 0; g < G; ++g) m_run[g] = kNegInf, l_run[g] = 0.f;

    for (int64_t ch = c0; ch < c1; ++ch) {
        const int64_t tbase = sh.first_token + ch * CHUNK + threadIdx.x;
        float sc[TPT][G];
        float cm[G];
#pragma unroll
        for (int g = 0; g < G; ++g) cm[g] = kNegInf;
#pragma unroll
        for (int r = 0; r < TPT; ++r) {
            const int64_t t = tbase + (int64_t)r * THREADS;
#pragma unroll
            for (int g = 0; g < G; ++g) sc[r][g] = kNegInf;
            if (t < sh.tokens) {
                uint32_t w[NS / 4];
                load_code_row<NS>(kb + (size_t)t * NS, w);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (g < gpb) {
                        const float *lg = lut + g * tab;
                        float a = 0.f;
#pragma unroll
                        for (int s = 0; s < NS; ++s) a += lg[s * kLutStride + code_at(w[s / 4], s % 4)];
                        sc[r][g] = a;
                        cm[g] = fmaxf(cm[g], a);
                    }
                }
            }
        }
        // block maximum of the chunk, per head (alternating buffers, so one
        // barrier per chunk suffices)
        float *rmax = red + (size_t)(ch & 1) * gpb * 32;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (g < gpb) {
                float m = cm[g];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                if (lane == 0) rmax[g * 32 + warp] = m;
            }
        }
        __syncthreads();
        bool rescale = false;
        float f[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            f[g] = 1.f;
            if (g < gpb) {
                float m = m_run[g];
#pragma unroll
                for (int k = 0; k < NW; ++k) m = fmaxf(m, rmax[g * 32 + k]);
                if (m > m_run[g] && m_run[g] > kNegInf) {
                    f[g] = exp2f(m_run[g] - m);
                    rescale = true;
                }
                l_run[g] *= f[g];
                m_run[g] = m;
            }
        }
        if (rescale) {  // same value in every thread of the block
#pragma unroll
            for (int g = 0; g < G; ++g)
                if (g < gpb && f[g] != 1.f)
                    for (int e = threadIdx.x; e < tab; e += THREADS) wsum[g * tab + e] *= f[g];
            __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < TPT; ++r) {
            const int64_t t = tbase + (int64_t)r * THREADS;
            if (t < sh.tokens) {
                uint32_t w[NS / 4];
                load_code_row<NS>(vb + (size_t)t * NS, w);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (g < gpb) {
                        const float p = exp2f(sc[r][g] - m_run[g]);
                        l_run[g] += p;
                        float *wg = wsum + g * tab;
#pragma unroll
                        for (int s = 0; s < NS; ++s) atomicAdd(&wg[s * kLutStride + code_at(w[s / 4], s % 4)], p);
                    }
                }
            }
        }
    }

    // ---- block sums, then out[g][s*SUB + i] = sum_c W[g][s][c] * Vcb[c][i]
    float *rsum = red + (size_t)2 * gpb * 32;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (g < gpb) {
            float l = l_run[g];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (lane == 0) rsum[g * 32 + warp] = l;
        }
    }
    __syncthreads();
    const int d = sh.head_dim;
    for (int e = threadIdx.x; e < gpb * d; e += THREADS) {
        const int g = e / d;
        const int j = e - g * d;
        const int s = j / sub, i = j - s * sub;
        const float *wg = wsum + g * tab + s * kLutStride;
        float acc = 0.f;
        for (int c = 0; c < nc; ++c) acc = fmaf(wg[c], to_f32(vc[(size_t)c * sub + i]), acc);
        float *pp = part + (((size_t)b * sh.heads_q + hq0 + g) * sh.splits + split) * (size_t)(d + 2);
        pp[2 + j] = acc;
        if (j == 0) {
            float l = 0.f;
            for (int k = 0; k < NW; ++k) l += rsum[g * 32 + k];
            pp[0] = m_run[g];
            pp[1] = l;
        }
    }
}

// Merge the partials: out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k.
// Launch: grid.x = n_rows (batch * heads_q), block = head_dim rounded up to 32.
template <typename T>
__global__ void attn_combine(const float *__restrict__ part, int64_t n_rows, int32_t head_dim,
                             int32_t splits, T *__restrict__ out)
{
    constexpr float kNegInf = -__builtin_huge_valf();
    const int64_t r = blockIdx.x;
    const int j = threadIdx.x;
    if (r >= n_rows || j >= head_dim) return;
    const float *pr = part + (size_t)r * splits * (head_dim + 2);
    float m = kNegInf;
    for (int k = 0; k < splits; ++k) m = fmaxf(m, pr[(size_t)k * (head_dim + 2)]);
    float l = 0.f, o = 0.f;
    if (m > kNegInf) {
        for (int k = 0; k < splits; ++k) {
            const float *pk = pr + (size_t)k * (head_dim + 2);
            const float f = exp2f(pk[0] - m);  // empty partials: 2^-inf = 0
            l = fmaf(f, pk[1], l);
            o = fmaf(f, pk[2 + j], o);
        }
    }
    from_f32(out[(size_t)r * head_dim + j], l > 0.f ? o / l : 0.f);
}

}  // namespace vqk
