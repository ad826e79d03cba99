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
// (2^(kappa x) = e^(scale x), so this is the usual softmax.)
//
// GB300 shape.  A block owns GPB query heads of one KV head (grouped-query
// attention: they share that head's codes and codebooks) and a run of
// CHUNK-token chunks of the cache, so each code row is read from HBM once for
// all GPB heads.  Per chunk:
//   phase A, one thread per token: the key code row is read with vector
//     loads and its score looked up for every head; the tables of up to four
//     heads are interleaved so one 16-byte shared load serves four heads, and
//     stored in slot order (attn_lut_q) so that the lanes of a wavefront never
//     meet in a bank, whatever the codes.  The chunk maximum raises the
//     running maximum (online softmax: the register accumulators are
//     rescaled), and the weights 2^(score - max) and the value code rows go
//     to shared memory;
//   phase B, one thread per (VW-column slice of the head, token stream): the
//     value rows are gathered from the value codebook in shared memory (fp32
//     for 8-column slices, else the input type widened in registers) and
//     accumulated with the weights of every head in registers (no atomics).
//     The codebook is held in bank-disjoint copies, sub-space s reading copy
//     s % ncopies, where a copy owns one (row bytes)-wide slot of every
//     128-byte line: the lanes that share a shared-memory wavefront
//     (consecutive sub-spaces of one token) never hit the same banks,
//     whatever the codes.
// The shared-memory gathers and the value FMAs bound this kernel, not HBM.
// Each block writes a partial (max, sum, out[D]) per query head to the
// caller's workspace; attn_combine merges the partials (flash-decoding).
// A code >= n_centroids reads a zero table entry and a zero value row (the
// decode of such a code is a zero row).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "vq_check.cuh"

namespace vqk {

constexpr int kLutStride = 256;  // table row stride (one entry per 8-bit code), in vectors
constexpr int kAttnThreads = 256;
constexpr int kAttnVw = 4;       // value columns per phase-B thread, at least

// Value columns per phase-B thread: a whole 16-byte piece of a 16-bit value
// row (8 columns) when the sub-space width allows, else 4.  Wider slices
// halve the gathers of codes and weights per value column.
__host__ __device__ constexpr int attn_vw(int sub, int elem) { return elem == 2 && sub % 8 == 0 ? 8 : kAttnVw; }

struct AttnShape {
    int64_t batch;
    int32_t heads_q, heads_kv, head_dim, sub_dim, n_centroids;
    int64_t tokens;       // cached tokens T
    int64_t first_token;  // first attended token (sliding window), else 0
    int64_t chunks;       // ceil((T - first_token) / CHUNK)
    int32_t splits;       // chunk runs per (batch, KV head, head group)
    float kappa;          // scale * log2(e)
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f32(float &d, float v) { d = v; }
__device__ __forceinline__ void from_f32(__half &d, float v) { d = __float2half_rn(v); }
__device__ __forceinline__ void from_f32(__nv_bfloat16 &d, float v) { d = __float2bfloat16_rn(v); }

// Tokens per phase-A thread and per chunk, by sub-space count.
__host__ __device__ constexpr int attn_tok_per_thread(int ns) { return ns <= 16 ? 2 : 1; }
__host__ __device__ constexpr int attn_chunk(int ns) { return kAttnThreads * attn_tok_per_thread(ns); }

// Value-codebook copies: rows of rb = sub * elem bytes; ncopies copies, each
// owning one rb-byte slot of every 128-byte line (one copy when rb >= 128).
__host__ __device__ inline int attn_vcopies(int sub, int elem)
{
    const int rb = sub * elem;
    return rb >= 128 ? 1 : 128 / rb;
}

// Bytes per element of the value-codebook copies for inputs of `elem` bytes:
// with 8-column slices (attn_vw) the 16-bit values are widened to fp32 once,
// when the copies are built, instead of at every gather.
__host__ __device__ constexpr int attn_vstore(int sub, int elem) { return attn_vw(sub, elem) == 8 ? 4 : elem; }

// Shared-memory layout, in order (bytes):
//   lut  [GPB / GP][NS / Q][kLutStride][Q][GP] fp32   GP = min(GPB, 4) heads per
//        vector, Q = attn_lut_q(GP, NS) sub-spaces side by side in a row;
//        after the last chunk it holds the per-stream accumulators
//        [streams][GPB][D] fp32 (the region is sized for both)
//   vcb  [256][ncopies] rows of `sub` elements (of T, fp32 with 8-column
//        slices: attn_vstore), zero past n_c
//   pw   [CHUNK][GPB] fp32                     weights of the chunk
//   red  [3][GPB][NW] fp32                     block maxima (two buffers), sums
//   vtile[CHUNK][NS] bytes                     value codes of the chunk
struct AttnSmem {
    size_t lut, vcb, pw, red, vtile, total;
};
__host__ __device__ inline AttnSmem attn_smem(int gpb, int ns, int sub, int elem)
{
    AttnSmem m;
    const int chunk = attn_chunk(ns);
    const size_t lut_bytes = (size_t)gpb * ns * kLutStride * 4;
    const size_t acc_bytes = (size_t)kAttnThreads * attn_vw(sub, elem) * gpb * 4;  // >= streams * GPB * D floats
    m.lut = 0;
    m.vcb = m.lut + (lut_bytes > acc_bytes ? lut_bytes : acc_bytes);
    const int ve = attn_vstore(sub, elem);
    m.pw = m.vcb + (size_t)256 * attn_vcopies(sub, ve) * sub * ve;
    m.pw = (m.pw + 15) / 16 * 16;
    m.red = m.pw + (size_t)chunk * gpb * 4;
    m.vtile = m.red + (size_t)3 * gpb * (kAttnThreads / 32) * 4;
    m.vtile = (m.vtile + 15) / 16 * 16;
    m.total = m.vtile + (size_t)chunk * ns;
    return m;
}

// Table layout.  Entry (s, code) of a pack sits in row (s / Q) * 256 + code,
// slot s % Q, a row being Q entries of GP floats (128 bytes when NS allows).
// Phase A thread with lane l visits the sub-spaces in the order
// s = i ^ (l % Q), i = 0, 1, ...: the Q lanes that share a shared-memory
// wavefront then read Q different slots, so their lookups never meet in a
// bank whatever the codes are.
__host__ __device__ constexpr int attn_lut_q(int gp, int ns) { return 32 / gp < ns ? 32 / gp : ns; }

// The code bytes of a token reordered so that byte i of `p` is byte i ^ lq of
// `w` (lq < Q <= NS; `sel` is the __byte_perm selector of lq % 4).
template <int NS, int Q>
__device__ __forceinline__ void xor_order_codes(const uint32_t (&w)[NS / 4], uint32_t (&p)[NS / 4],
                                                uint32_t lq, uint32_t sel)
{
#pragma unroll
    for (int m = 0; m < NS / 4; ++m) p[m] = w[m];
#pragma unroll
    for (int bit = 0; (4 << bit) < Q; ++bit) {  // word index: m -> m ^ (lq / 4)
        const bool flip = (lq >> (2 + bit)) & 1u;
#pragma unroll
        for (int m = 0; m < NS / 4; ++m) {
            if (m & (1 << bit)) continue;
            const uint32_t x = p[m], y = p[m | (1 << bit)];
            p[m] = flip ? y : x;
            p[m | (1 << bit)] = flip ? x : y;
        }
    }
#pragma unroll
    for (int m = 0; m < NS / 4; ++m) p[m] = __byte_perm(p[m], 0u, sel);  // byte: t -> t ^ (lq % 4)
}

// Four consecutive elements of a value row in shared memory, widened.
__device__ __forceinline__ float4 load4_f32(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4_f32(const __half *p)
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 load4_f32(const __nv_bfloat16 *p)
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// Two 16-bit elements packed in a word, widened (element 0 in the low half).
__device__ __forceinline__ float2 pair_f32(uint32_t w, const __half *)
{
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
__device__ __forceinline__ float2 pair_f32(uint32_t w, const __nv_bfloat16 *)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Eight consecutive fp32 elements of a value row in shared memory as column
// pairs, the half h (columns 4h .. 4h+3) first: r[0], r[1] hold columns
// 4h .. 4h+3, r[2], r[3] the other four.
__device__ __forceinline__ void load_row(const float *p, int h, float2 (&r)[4])
{
    const float4 a = *reinterpret_cast<const float4 *>(p + 4 * h);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4 - 4 * h);
    r[0] = make_float2(a.x, a.y), r[1] = make_float2(a.z, a.w);
    r[2] = make_float2(b.x, b.y), r[3] = make_float2(b.z, b.w);
}

// Four consecutive elements of a value row in shared memory (the input
// type), widened, as column pairs (4-column slices; 8-column slices read the
// fp32 copies through the overload above).
template <int VW, typename T>
__device__ __forceinline__ void load_row(const T *p, float2 (&r)[VW / 2])
{
    static_assert(VW == 4, "4-column slices");
    const float4 a = load4_f32(p);
    r[0] = make_float2(a.x, a.y), r[1] = make_float2(a.z, a.w);
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

template <int NS>
__device__ __forceinline__ void store_code_row(uint8_t *p, const uint32_t (&w)[NS / 4])
{
    if constexpr (NS % 16 == 0) {
#pragma unroll
        for (int k = 0; k < NS / 16; ++k)
            reinterpret_cast<uint4 *>(p)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    } else if constexpr (NS % 8 == 0) {
#pragma unroll
        for (int k = 0; k < NS / 8; ++k) reinterpret_cast<uint2 *>(p)[k] = make_uint2(w[2 * k], w[2 * k + 1]);
    } else {
#pragma unroll
        for (int k = 0; k < NS / 4; ++k) reinterpret_cast<uint32_t *>(p)[k] = w[k];
    }
}

__device__ __forceinline__ uint32_t code_at(uint32_t w, int k) { return (w >> (8 * k)) & 0xffu; }

// (a.x * b + c.x, a.y * b + c.y) as one packed f32x2 FMA, each lane rounded
// once as fmaf would.
__device__ __forceinline__ float2 fma2_bcast(float2 a, float b, float2 c)
{
    return __ffma2_rn(a, make_float2(b, b), c);
}

// GP consecutive floats from shared memory (GP = 1, 2 or 4, aligned).
template <int GP>
__device__ __forceinline__ void load_vec(const float *p, float (&v)[GP])
{
    if constexpr (GP == 4) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w;
    } else if constexpr (GP == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(p);
        v[0] = a.x, v[1] = a.y;
    } else {
        v[0] = *p;
    }
}

// Warp maxima of GPB values per lane, with log2(GPB) exchanges that halve
// the values a lane carries (lanes with bit 16 >> r set keep the upper half
// in round r) and plain exchanges after: the lanes l with
// l % (32 / GPB) == 0 return the warp's maximum of value `head`.
template <int GPB>
__device__ __forceinline__ float warp_max_heads(const float (&v)[GPB], int lane, int &head)
{
    float w[GPB];
#pragma unroll
    for (int g = 0; g < GPB; ++g) w[g] = v[g];
    head = 0;
#pragma unroll
    for (int r = 0; (1 << r) < GPB; ++r) {
        const int off = 16 >> r, half = GPB >> (r + 1);
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float send = upper ? w[k] : w[k + half];
            const float keep = upper ? w[k + half] : w[k];
            w[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, off));
        }
        head += upper ? half : 0;
    }
#pragma unroll
    for (int off = 32 / GPB / 2; off > 0; off >>= 1) w[0] = fmaxf(w[0], __shfl_xor_sync(0xffffffffu, w[0], off));
    return w[0];
}

// Block maxima of the GPB heads from the NW warp maxima rmax[g * NW + w]:
// lane l reads entries l and l + 32, groups of NW lanes reduce, and every
// lane takes head g's maximum from lane (g % (32 / NW)) * NW.
template <int GPB, int NW>
__device__ __forceinline__ void block_max_heads(const float *rmax, const float *red, uint64_t red_floats,
                                                int lane, float (&bm)[GPB])
{
    constexpr float kNegInf = -__builtin_huge_valf();
    constexpr int ROUNDS = (GPB * NW + 31) / 32;
    constexpr int HPR = 32 / NW;  // heads per round of 32 entries
    static_assert(32 % NW == 0, "whole heads per round");
    float v[ROUNDS];
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int e = r * 32 + lane;
        v[r] = e < GPB * NW && VQ_SPAN(rmax + e, 1, red, red_floats) ? rmax[e] : kNegInf;
#pragma unroll
        for (int off = NW / 2; off > 0; off >>= 1) v[r] = fmaxf(v[r], __shfl_xor_sync(0xffffffffu, v[r], off));
    }
#pragma unroll
    for (int g = 0; g < GPB; ++g) bm[g] = __shfl_sync(0xffffffffu, v[g / HPR], (g % HPR) * NW);
}

// Scores of one token for the block's GPB heads (phase A): its key code
// row `wk` (NS bytes), looked up in the slot-ordered tables, sub-spaces in
// the order i ^ lq (lq = lane % Q; lq_sel the byte selector of lq % 4).
template <int NS, int GPB>
__device__ __forceinline__ void attn_token_scores(const uint32_t (&wk)[NS / 4], const float *lut,
                                                  uint64_t lut_floats, uint32_t lq, uint32_t lq_sel,
                                                  float (&a)[GPB])
{
    constexpr int GP = GPB < 4 ? GPB : 4;
    constexpr int NPACK = GPB / GP;
    constexpr int Q = attn_lut_q(GP, NS);
    const int lq_f = (int)lq * GP;
    (void)lut_floats;
#pragma unroll
    for (int g = 0; g < GPB; ++g) a[g] = 0.f;
    uint32_t wq[NS / 4];  // byte i = code of sub-space i ^ lq
    xor_order_codes<NS, Q>(wk, wq, lq, lq_sel);
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int code = (int)code_at(wq[i / 4], i % 4);
        // slot (i % Q) ^ lq of row (i / Q) * 256 + code
        const int slot_f = ((i % Q) * GP) ^ lq_f;
#pragma unroll
        for (int pk = 0; pk < NPACK; ++pk) {
            float v[GP];
            const float *src =
                lut + ((size_t)pk * NS + (i / Q) * Q) * kLutStride * GP + code * (Q * GP) + slot_f;
            if (VQ_VSPAN(src, GP, lut, lut_floats, GP * 4)) {
                load_vec<GP>(src, v);
            } else {
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) v[gi] = 0.f;
            }
            if constexpr (GP >= 2) {  // head pairs as packed adds
#pragma unroll
                for (int gi = 0; gi < GP; gi += 2) {
                    const float2 t2 = __fadd2_rn(make_float2(a[pk * GP + gi], a[pk * GP + gi + 1]),
                                                 make_float2(v[gi], v[gi + 1]));
                    a[pk * GP + gi] = t2.x, a[pk * GP + gi + 1] = t2.y;
                }
            } else {
                a[pk] += v[0];
            }
        }
    }
}

// The block's tables and value-codebook copies (attn_partial):
// stage the queries of heads hq0 .. hq0 + GPB - 1 of batch row b, build the
// GP-interleaved, slot-ordered key tables in `lut` (lut_floats floats) and
// the value codebook's `ncopies` copies in `vcs` as VT (T, or fp32 for
// 16-bit T) (a region of region_bytes bytes, vcs_elems elements used).  kc, vc: the KV head's codebooks.  Ends
// with a block barrier.
template <typename T, typename VT, int NS, int GPB, int THREADS>
__device__ __forceinline__ void attn_setup(const T *__restrict__ q, const T *__restrict__ kcb,
                                           const T *__restrict__ vcb, const AttnShape &sh, int64_t b,
                                           int hq0, const T *kc, const T *vc, float *lut,
                                           uint64_t lut_floats, VT *vcs, uint64_t vcs_elems,
                                           uint64_t region_bytes, int ncopies)
{
    constexpr int GP = GPB < 4 ? GPB : 4;
    constexpr int NPACK = GPB / GP;
    constexpr int Q = attn_lut_q(GP, NS);
    const int sub = sh.sub_dim;
    const int d = sh.head_dim;
    const int nc = sh.n_centroids;
    const int64_t nq_elems = sh.batch * sh.heads_q * d;
    const int64_t ncb_elems = (int64_t)sh.heads_kv * nc * sub;
    (void)nq_elems, (void)ncb_elems, (void)kcb, (void)vcb;

    // ---- the block's queries, widened to fp32 and transposed, staged in
    // the value-codebook region, which is not in use yet: element s * sub + i
    // of head g at qT[s * qs_stride + i * GPB + g].  The 4-float pad per
    // sub-space puts the rows that the lanes of a wavefront read (different
    // sub-spaces, below) in different banks.  At most 17 KiB; the region
    // holds at least 18 KiB (attn_plan checks).
    float *qT = reinterpret_cast<float *>(vcs);
    const int qs_stride = sub * GPB + 4;
    const uint64_t qT_floats = (uint64_t)NS * qs_stride;
    for (int e = threadIdx.x; e < GPB * d; e += THREADS) {
        const int g = e / d, j = e - g * d;
        const int sj = j / sub, ij = j - sj * sub;
        const T *src = q + ((size_t)b * sh.heads_q + hq0 + g) * d + j;
        float *dst = qT + (size_t)sj * qs_stride + (size_t)ij * GPB + g;
        if (VQ_SPAN(dst, 1, qT, region_bytes / 4))
            *dst = VQ_SPAN(src, 1, q, nq_elems) ? to_f32(*src) : 0.f;
    }
    __syncthreads();

    // ---- tables (kappa folded in, zero past n_centroids): thread c owns
    // centroid c and writes the GP heads of a pack as one vector, visiting
    // the sub-spaces in the order i ^ (c % Q) so that the stores of a warp
    // spread over the slots.  A 16-byte codebook row is read once into
    // registers; other widths are read element by element.
    constexpr int KR = 16 / (int)sizeof(T);  // elements in a 16-byte row
    const bool row16 = sub == KR && ((uintptr_t)kc & 15u) == 0;
    for (int c = threadIdx.x; c < kLutStride; c += THREADS) {
        const T *cv = kc + (size_t)c * sub;
        const bool live = c < nc && VQ_SPAN(cv, sub, kcb, ncb_elems);
        float kr[KR];
#pragma unroll
        for (int i = 0; i < KR; ++i) kr[i] = 0.f;
        if (row16 && live && VQ_VSPAN(cv, KR, kcb, ncb_elems, 16)) {
            const uint4 u = *reinterpret_cast<const uint4 *>(cv);
            const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if constexpr (sizeof(T) == 4) {
                    kr[k] = __uint_as_float(uw[k]);
                } else {
                    const float2 f = pair_f32(uw[k], cv);
                    kr[2 * k] = f.x, kr[2 * k + 1] = f.y;
                }
            }
        }
#pragma unroll
        for (int pk = 0; pk < NPACK; ++pk) {
            for (int si = 0; si < NS; ++si) {
                const int s = si ^ (c & (Q - 1));
                const float *qs = qT + (size_t)s * qs_stride + pk * GP;  // query element s * sub
                float acc[GP];
#pragma unroll
                for (int gi = 0; gi < GP; ++gi) acc[gi] = 0.f;
                if (live) {
                    if (row16) {
#pragma unroll
                        for (int i = 0; i < KR; ++i) {
                            float qv[GP];
                            if (VQ_VSPAN(qs + (size_t)i * GPB, GP, qT, qT_floats, GP * 4)) {
                                load_vec<GP>(qs + (size_t)i * GPB, qv);
#pragma unroll
                                for (int gi = 0; gi < GP; ++gi) acc[gi] = fmaf(qv[gi], kr[i], acc[gi]);
                            }
                        }
                    } else {
                        for (int i = 0; i < sub; ++i) {
                            const float kv = to_f32(cv[i]);
                            float qv[GP];
                            if (VQ_VSPAN(qs + (size_t)i * GPB, GP, qT, qT_floats, GP * 4)) {
                                load_vec<GP>(qs + (size_t)i * GPB, qv);
#pragma unroll
                                for (int gi = 0; gi < GP; ++gi) acc[gi] = fmaf(qv[gi], kv, acc[gi]);
                            }
                        }
                    }
                }
                float *dst = lut + (((size_t)pk * NS + (s / Q) * Q) * kLutStride + (size_t)c * Q + s % Q) * GP;
                if (VQ_SPAN(dst, GP, lut, lut_floats)) {
#pragma unroll
                    for (int gi = 0; gi < GP; ++gi) dst[gi] = acc[gi] * sh.kappa;
                }
            }
        }
    }
    __syncthreads();  // the staged queries are read no more

    // ---- the value codebook in its bank-disjoint copies (zero past
    // n_centroids): 16-byte pieces of the rows where they allow, each stored
    // (widened to fp32 when VT is) to every copy, starting at copy
    // c % ncopies so that a warp's stores spread over the copies; else
    // element by element
    const int rbytes = sub * (int)sizeof(T);
    if (rbytes % 16 == 0 && ((uintptr_t)vc & 15u) == 0) {
        const int pieces = rbytes / 16;
        for (int e = threadIdx.x; e < kLutStride * pieces; e += THREADS) {
            const int c = e / pieces, w = e - c * pieces;
            const T *src = vc + (size_t)c * sub + (size_t)w * KR;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (c < nc && VQ_VSPAN(src, KR, vcb, ncb_elems, 16)) v = *reinterpret_cast<const uint4 *>(src);
            int j = c % ncopies;
            for (int k = 0; k < ncopies; ++k) {
                VT *dst = vcs + ((size_t)c * ncopies + j) * sub + (size_t)w * KR;
                if (VQ_VSPAN(dst, KR, vcs, vcs_elems, 16)) {
                    if constexpr (std::is_same<VT, T>::value) {
                        *reinterpret_cast<uint4 *>(dst) = v;
                    } else {  // eight 16-bit values to fp32
                        const float2 f0 = pair_f32(v.x, src), f1 = pair_f32(v.y, src);
                        const float2 f2 = pair_f32(v.z, src), f3 = pair_f32(v.w, src);
                        reinterpret_cast<float4 *>(dst)[0] = make_float4(f0.x, f0.y, f1.x, f1.y);
                        reinterpret_cast<float4 *>(dst)[1] = make_float4(f2.x, f2.y, f3.x, f3.y);
                    }
                }
                j = j + 1 == ncopies ? 0 : j + 1;
            }
        }
    } else {
        for (int c = threadIdx.x; c < kLutStride; c += THREADS) {
            for (int i = 0; i < sub; ++i) {
                const T v = c < nc && VQ_SPAN(vc + (size_t)c * sub + i, 1, vcb, ncb_elems) ? vc[(size_t)c * sub + i] : T(0.f);
                for (int j = 0; j < ncopies; ++j)
                    if (VQ_SPAN(vcs + ((size_t)c * ncopies + j) * sub + i, 1, vcs, vcs_elems)) {
                        if constexpr (std::is_same<VT, T>::value) {
                            vcs[((size_t)c * ncopies + j) * sub + i] = v;
                        } else {
                            vcs[((size_t)c * ncopies + j) * sub + i] = to_f32(v);
                        }
                    }
            }
        }
    }
    __syncthreads();
}

// Launch: grid.x = batch * heads_kv * (heads_q / heads_kv / GPB) * splits,
// block = kAttnThreads, dynamic shared memory attn_smem(GPB, NS, SUB, sizeof(T)).total,
// VW = attn_vw(SUB, sizeof(T)).
// NS = head_dim / sub_dim in {4, 8, 16, 32, 64}; sub_dim % 4 == 0; code rows
// are NS bytes apart and the code arrays aligned to min(NS, 16) bytes.
// Partial of (b, hq, split) at part[((b * heads_q + hq) * splits + split) *
// (D + 2)]: {0: max (log2 domain), 1: sum, 2..: unnormalised out}.
template <typename T, int NS, int GPB, int VW>
__global__ void __launch_bounds__(kAttnThreads)
    attn_partial(const T *__restrict__ q, const uint8_t *__restrict__ kcodes,
                 const T *__restrict__ kcb, const uint8_t *__restrict__ vcodes,
                 const T *__restrict__ vcb, AttnShape sh, float *__restrict__ part)
{
    constexpr int THREADS = kAttnThreads;
    constexpr int TPT = attn_tok_per_thread(NS);
    constexpr int CHUNK = attn_chunk(NS);
    constexpr int GP = GPB < 4 ? GPB : 4;
    constexpr int NPACK = GPB / GP;
    constexpr int Q = attn_lut_q(GP, NS);
    static_assert(NS % Q == 0 && (Q & (Q - 1)) == 0, "table rows hold a power-of-two divisor of NS");
    constexpr int NW = THREADS / 32;
    constexpr float kNegInf = -__builtin_huge_valf();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int sub = sh.sub_dim;
    const int d = sh.head_dim;
    const int nc = sh.n_centroids;
    const AttnSmem lay = attn_smem(GPB, NS, sub, (int)sizeof(T));
    using VT = typename std::conditional<VW == 8, float, T>::type;  // value-copy element (attn_vstore)
    const int ncopies = attn_vcopies(sub, (int)sizeof(VT));
    float *lut = reinterpret_cast<float *>(smem_raw + lay.lut);
    VT *vcs = reinterpret_cast<VT *>(smem_raw + lay.vcb);
    float *pw = reinterpret_cast<float *>(smem_raw + lay.pw);
    float *red = reinterpret_cast<float *>(smem_raw + lay.red);
    uint8_t *vtile = smem_raw + lay.vtile;

    const int qpk = sh.heads_q / sh.heads_kv;  // query heads per KV head
    const int hgroups = qpk / GPB;
    int64_t bid = blockIdx.x;
    const int split = (int)(bid % sh.splits);
    bid /= sh.splits;
    const int hg = (int)(bid % hgroups);
    bid /= hgroups;
    const int hkv = (int)(bid % sh.heads_kv);
    const int64_t b = bid / sh.heads_kv;
    const int hq0 = hkv * qpk + hg * GPB;

    const T *kc = kcb + (size_t)hkv * nc * sub;
    const T *vc = vcb + (size_t)hkv * nc * sub;
    const size_t cache_off = ((size_t)b * sh.heads_kv + hkv) * (size_t)sh.tokens * NS;
    const uint8_t *kb = kcodes + cache_off;
    const uint8_t *vb = vcodes + cache_off;

    // buffer extents, for the checked build's bounds checks (vq_check.cuh)
    const int64_t ncodes = sh.batch * sh.heads_kv * sh.tokens * NS;
    const int64_t npart = sh.batch * sh.heads_q * sh.splits * (int64_t)(d + 2);
    const uint64_t lut_floats = (lay.vcb - lay.lut) / 4, vcs_elems = (uint64_t)256 * ncopies * sub;
    const uint64_t pw_floats = (uint64_t)CHUNK * GPB, red_floats = (uint64_t)3 * GPB * NW;
    constexpr uint32_t kCodeAlign = NS < 16 ? NS : 16;  // load_code_row, store_code_row
    if constexpr (kChecked) {
        // the layout inside the launch's shared memory and the block inside
        // the grid: else the block does nothing
        if (!dyn_smem_ok(smem_raw, lay.total, 16) || !index_ok(b, sh.batch) || vcs_elems * sizeof(VT) > lay.pw - lay.vcb ||
            attn_vw(sub, (int)sizeof(T)) != VW)
            return;  // block-uniform
    }

    attn_setup<T, VT, NS, GPB, THREADS>(q, kcb, vcb, sh, b, hq0, kc, vc, lut, lut_floats, vcs, vcs_elems,
                                    lay.pw - lay.vcb, ncopies);

    // phase-B role: VW-column slice `col` (columns col*VW .. col*VW+VW-1 of
    // the head, inside one sub-space), token stream `stream` of `streams`
    const int ncols = d / VW;
    const int streams = THREADS / ncols;
    const int col = threadIdx.x % ncols;
    const int stream = threadIdx.x / ncols;
    const bool b_active = stream < streams;
    const int bs = (col * VW) / sub;            // sub-space of the slice
    const int bi = (col * VW) - bs * sub;       // first element in the row
    // this slice's columns in copy bs % ncopies of code 0; code c adds c rows
    const VT *vrow0 = vcs + (size_t)(bs % ncopies) * sub + bi;
    const size_t vstride = (size_t)ncopies * sub;
    // fp32 rows: the two slices that share a copy in one wavefront read
    // its two 16-byte halves in opposite orders (load_row)
    const int vh = (bs / ncopies) & 1;
    float2 acc[GPB][VW / 2];  // column pairs (0, 1), (2, 3), ... of the slice
#pragma unroll
    for (int g = 0; g < GPB; ++g)
#pragma unroll
        for (int i = 0; i < VW / 2; ++i) acc[g][i] = make_float2(0.f, 0.f);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // phase-A sub-space order (see attn_lut_q)
    const uint32_t lq = (uint32_t)lane & (Q - 1);
    const uint32_t lq_sel = 0x3210u ^ ((lq & 3u) * 0x1111u);
    float m_run[GPB], l_run[GPB];
#pragma unroll
    for (int g = 0; g < GPB; ++g) m_run[g] = kNegInf, l_run[g] = 0.f;

    const int64_t c0 = sh.chunks * split / sh.splits;
    const int64_t c1 = sh.chunks * (split + 1) / sh.splits;
    // code rows of this thread's phase-A tokens, loaded one chunk ahead
    uint32_t wk[TPT][NS / 4], wv[TPT][NS / 4];
    auto load_rows = [&](int64_t ch) {
        const int64_t tb = sh.first_token + ch * CHUNK + threadIdx.x;
#pragma unroll
        for (int r = 0; r < TPT; ++r) {
            const int64_t t = tb + (int64_t)r * THREADS;
            if (t < sh.tokens && VQ_VSPAN(kb + (size_t)t * NS, NS, kcodes, ncodes, kCodeAlign) &&
                VQ_VSPAN(vb + (size_t)t * NS, NS, vcodes, ncodes, kCodeAlign)) {
                load_code_row<NS>(kb + (size_t)t * NS, wk[r]);
                load_code_row<NS>(vb + (size_t)t * NS, wv[r]);
            }
        }
    };
    if (c0 < c1) load_rows(c0);
    for (int64_t ch = c0; ch < c1; ++ch) {
        const int64_t tbase = sh.first_token + ch * CHUNK;
        // ---- phase A: scores of TPT tokens per thread
        float sc[TPT][GPB];
        float cm[GPB];
#pragma unroll
        for (int g = 0; g < GPB; ++g) cm[g] = kNegInf;
#pragma unroll
        for (int r = 0; r < TPT; ++r) {
            const int64_t t = tbase + r * THREADS + threadIdx.x;
#pragma unroll
            for (int g = 0; g < GPB; ++g) sc[r][g] = kNegInf;
            if (t < sh.tokens) {
                float a[GPB];
                attn_token_scores<NS, GPB>(wk[r], lut, lut_floats, lq, lq_sel, a);
#pragma unroll
                for (int g = 0; g < GPB; ++g) {
                    sc[r][g] = a[g];
                    cm[g] = fmaxf(cm[g], a[g]);
                }
            }
        }
        // block maximum of the chunk (alternating buffers).  This barrier
        // also ends the previous chunk's phase B, so the weights and value
        // codes below may be overwritten after it.
        float *rmax = red + (size_t)(ch & 1) * GPB * NW;
        {
            int head;
            const float m = warp_max_heads<GPB>(cm, lane, head);
            if ((lane & (32 / GPB - 1)) == 0 && VQ_SPAN(rmax + head * NW + warp, 1, red, red_floats))
                rmax[head * NW + warp] = m;
        }
        __syncthreads();
        float bm[GPB];
        block_max_heads<GPB, NW>(rmax, red, red_floats, lane, bm);
#pragma unroll
        for (int g = 0; g < GPB; ++g) {
            const float m = fmaxf(m_run[g], bm[g]);
            if (m > m_run[g] && m_run[g] > kNegInf) {  // rescale what is accumulated
                const float f = exp2f(m_run[g] - m);
                l_run[g] *= f;
#pragma unroll
                for (int i = 0; i < VW / 2; ++i) acc[g][i] = make_float2(acc[g][i].x * f, acc[g][i].y * f);
            }
            m_run[g] = m;
        }
#pragma unroll
        for (int r = 0; r < TPT; ++r) {
            const int tl = r * THREADS + threadIdx.x;
            float p[GPB];
#pragma unroll
            for (int g = 0; g < GPB; ++g) {
                // tokens past the end: sc = -inf, weight 0
                p[g] = sc[r][g] == kNegInf ? 0.f : exp2f(sc[r][g] - m_run[g]);
                l_run[g] += p[g];
            }
#pragma unroll
            for (int pk = 0; pk < NPACK; ++pk) {
                float *dst = pw + (size_t)tl * GPB + pk * GP;
                if (!VQ_VSPAN(dst, GP, pw, pw_floats, GP * 4)) continue;
                if constexpr (GP == 4) {
                    *reinterpret_cast<float4 *>(dst) = make_float4(p[pk * 4], p[pk * 4 + 1], p[pk * 4 + 2], p[pk * 4 + 3]);
                } else if constexpr (GP == 2) {
                    *reinterpret_cast<float2 *>(dst) = make_float2(p[pk * 2], p[pk * 2 + 1]);
                } else {
                    dst[0] = p[pk];
                }
            }
            if (tbase + tl < sh.tokens && VQ_VSPAN(vtile + (size_t)tl * NS, NS, vtile, (uint64_t)CHUNK * NS, kCodeAlign))
                store_code_row<NS>(vtile + (size_t)tl * NS, wv[r]);
        }
        if (ch + 1 < c1) load_rows(ch + 1);  // in flight during phase B
        __syncthreads();
        // ---- phase B: weighted value rows, accumulated in registers
        const int64_t n_in = sh.tokens - tbase;
        const int n_chunk = n_in < CHUNK ? (int)n_in : CHUNK;
        if (b_active) {
            constexpr int U = 4;
            int tl = stream;
            for (; tl + (U - 1) * streams < n_chunk; tl += U * streams) {
                int code[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    code[u] = VQ_SPAN(vtile + (size_t)(tl + u * streams) * NS + bs, 1, vtile, (uint64_t)CHUNK * NS)
                                  ? vtile[(size_t)(tl + u * streams) * NS + bs] : 0;
                float2 row[U][VW / 2];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (VQ_VSPAN(vrow0 + (size_t)code[u] * vstride, VW, vcs, vcs_elems, VW == 8 ? 16 : VW * sizeof(T))) {
                        if constexpr (VW == 8)
                            load_row(vrow0 + (size_t)code[u] * vstride, vh, row[u]);
                        else
                            load_row<VW>(vrow0 + (size_t)code[u] * vstride, row[u]);
                    } else {
#pragma unroll
                        for (int i = 0; i < VW / 2; ++i) row[u][i] = make_float2(0.f, 0.f);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    float p[GPB];
#pragma unroll
                    for (int pk = 0; pk < NPACK; ++pk) {
                        float v[GP];
                        if (!VQ_VSPAN(pw + (size_t)(tl + u * streams) * GPB + pk * GP, GP, pw, pw_floats, GP * 4)) {
#pragma unroll
                            for (int gi = 0; gi < GP; ++gi) p[pk * GP + gi] = 0.f;
                            continue;
                        }
                        load_vec<GP>(pw + (size_t)(tl + u * streams) * GPB + pk * GP, v);
#pragma unroll
                        for (int gi = 0; gi < GP; ++gi) p[pk * GP + gi] = v[gi];
                    }
#pragma unroll
                    for (int g = 0; g < GPB; ++g)
#pragma unroll
                        for (int i = 0; i < VW / 2; ++i) acc[g][i] = fma2_bcast(row[u][i], p[g], acc[g][i]);
                }
            }
            for (; tl < n_chunk; tl += streams) {
                const int code = VQ_SPAN(vtile + (size_t)tl * NS + bs, 1, vtile, (uint64_t)CHUNK * NS)
                                     ? vtile[(size_t)tl * NS + bs] : 0;
                float2 row[VW / 2];
                if (VQ_VSPAN(vrow0 + (size_t)code * vstride, VW, vcs, vcs_elems, VW == 8 ? 16 : VW * sizeof(T))) {
                    if constexpr (VW == 8)
                        load_row(vrow0 + (size_t)code * vstride, vh, row);
                    else
                        load_row<VW>(vrow0 + (size_t)code * vstride, row);
                } else {
#pragma unroll
                    for (int i = 0; i < VW / 2; ++i) row[i] = make_float2(0.f, 0.f);
                }
                float p[GPB];
#pragma unroll
                for (int pk = 0; pk < NPACK; ++pk) {
                    float v[GP];
                    if (!VQ_VSPAN(pw + (size_t)tl * GPB + pk * GP, GP, pw, pw_floats, GP * 4)) {
#pragma unroll
                        for (int gi = 0; gi < GP; ++gi) p[pk * GP + gi] = 0.f;
                        continue;
                    }
                    load_vec<GP>(pw + (size_t)tl * GPB + pk * GP, v);
#pragma unroll
                    for (int gi = 0; gi < GP; ++gi) p[pk * GP + gi] = v[gi];
                }
#pragma unroll
                for (int g = 0; g < GPB; ++g)
#pragma unroll
                    for (int i = 0; i < VW / 2; ++i) acc[g][i] = fma2_bcast(row[i], p[g], acc[g][i]);
            }
        }
    }
    __syncthreads();  // the tables are reused below

    // the dependent merge kernel may be scheduled from here on; it waits for
    // this whole grid before it reads any partial
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- block sums and the merge of the token streams
    float *rsum = red + (size_t)2 * GPB * NW;
#pragma unroll
    for (int g = 0; g < GPB; ++g) {
        float l = l_run[g];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0 && VQ_SPAN(rsum + g * NW + warp, 1, red, red_floats)) rsum[g * NW + warp] = l;
    }
    float *accs = lut;  // [streams][GPB][D]; the tables are no longer read
    if (b_active) {
#pragma unroll
        for (int g = 0; g < GPB; ++g)
            if (VQ_VSPAN(accs + ((size_t)stream * GPB + g) * d + col * VW, VW, lut, lut_floats, 16)) {
#pragma unroll
                for (int i = 0; i < VW / 4; ++i) {
                    // with fp32 rows, acc[g][0..1] hold columns 4 vh .. 4 vh + 3
                    const int slot = VW == 8 ? i ^ vh : i;
                    reinterpret_cast<float4 *>(accs + ((size_t)stream * GPB + g) * d + col * VW)[slot] =
                        make_float4(acc[g][2 * i].x, acc[g][2 * i].y, acc[g][2 * i + 1].x, acc[g][2 * i + 1].y);
                }
            }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < GPB * d; e += THREADS) {
        const int g = e / d;
        const int j = e - g * d;
        float o = 0.f;
        for (int k = 0; k < streams; ++k)
            if (VQ_SPAN(accs + ((size_t)k * GPB + g) * d + j, 1, lut, lut_floats)) o += accs[((size_t)k * GPB + g) * d + j];
        float *pp = part + (((size_t)b * sh.heads_q + hq0 + g) * sh.splits + split) * (size_t)(d + 2);
        if (!VQ_SPAN(pp, d + 2, part, npart)) continue;
        pp[2 + j] = o;
        if (j == 0) {
            float l = 0.f, m = m_run[0];
            for (int k = 0; k < NW; ++k)
                if (VQ_SPAN(rsum + g * NW + k, 1, red, red_floats)) l += rsum[g * NW + k];
#pragma unroll
            for (int gg = 1; gg < GPB; ++gg)
                if (gg == g) m = m_run[gg];  // static register index
            pp[0] = m;
            pp[1] = l;
        }
    }
}

// Merge the partials: out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k.
// Launch: grid.x = n_rows (batch * heads_q), block = head_dim rounded up to
// 32, after attn_partial on the same stream, as its programmatic dependent
// (or plainly: the wait below then returns at once).
template <typename T>
__global__ void attn_combine(const float *__restrict__ part, int64_t n_rows, int32_t head_dim,
                             int32_t splits, T *__restrict__ out)
{
    constexpr float kNegInf = -__builtin_huge_valf();
    const int64_t r = blockIdx.x;
    const int j = threadIdx.x;
    // launched as a programmatic dependent of attn_partial: wait until that
    // grid has completed and its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (r >= n_rows || j >= head_dim) return;
    const float *pr = part + (size_t)r * splits * (head_dim + 2);
    if (!VQ_SPAN(pr, (int64_t)splits * (head_dim + 2), part, n_rows * splits * (int64_t)(head_dim + 2)) ||
        !VQ_SPAN(out + (size_t)r * head_dim + j, 1, out, n_rows * head_dim))
        return;
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
