// vq_scalar.cuh -- sibling encoders on the same nearest-centroid rule (the
// page of five hand-tuned Metal compute kernels for TurboQuant, sections
// "Kernel 2: Scalar Quantize / Dequantize" and "Kernel 3: Fused Hadamard +
// Quantize"):
//   scalar quantize   idx[e] = argmin_j fl(fl(float(x[e]) - c[j])^2), strict
//                     "<" over ascending j from (+inf, 0), one fp32 codebook;
//   Hadamard rotate   v = float(x) * diag; butterfly passes stride 1, 2, ...,
//                     D/2: (lo, hi) -> (lo + hi, lo - hi); y = v * scale;
//   fused quantize    idx = scalar quantize of y.
// Every operation is an explicitly rounded fp32 intrinsic (or packed f32x2
// form, each lane rounded alike), arranged so that no compiler contraction
// can change a result.
//
// GB300 shape.  fp16 keys against 2, 4, 8 or 16 centroids take
// scalar_bucket: each block builds, from the codebook's cut points, one entry
// per 10-bit prefix of the fp16 pattern (the codes on either side of the
// bucket's one change of code, or a flag) and copies the entries once per
// shared-memory bank, so the pass is a coalesced 2-byte-in / 1-byte-out
// stream with one conflict-free shared-memory lookup per element.  Other
// 16-bit inputs have only 65,536 values too: scalar_table evaluates the
// formula once for each bit pattern into a 64 KiB table (the caller's
// workspace), and scalar_lookup stages that table in shared memory and looks
// every element up there.  Both are bit-identical to the scan.  Other inputs
// use scalar_scan: codebooks of 2, 4, 8 or 16 finite entries go
// through a packed register scan (distances in f32x2 pairs, their least by a
// min3 tree, the lowest index holding it from sign bits), others through a
// sorted view of the codebook with the scan as fallback.  The rotation
// spreads each row over up to 32 lanes: a lane holds E contiguous elements
// (at least 8 when x is aligned for it), so butterfly strides below E stay
// in registers and larger ones are shfl.xor exchanges; no shared memory and
// no barriers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "vq_check.cuh"

namespace vqs {

__device__ __forceinline__ float widen16(uint16_t bits, bool bf16)
{
    return bf16 ? __uint_as_float((uint32_t)bits << 16) : __half2float(__ushort_as_half(bits));
}
__device__ __forceinline__ float widen_elem(float v) { return v; }
__device__ __forceinline__ float widen_elem(__half v) { return __half2float(v); }
__device__ __forceinline__ float widen_elem(__nv_bfloat16 v) { return __bfloat162float(v); }

// The nearest-centroid rule for one fp32 value, codebook c[0..n_c) in shared
// memory (every lane reads the same entry: broadcast).
__device__ __forceinline__ uint32_t nearest(float val, const float *c, int n_c)
{
    float best_dist = __int_as_float(0x7f800000);
    uint32_t best = 0;
    for (int j = 0; j < n_c; ++j) {
        const float d = __fsub_rn(val, c[j]);
        const float dist = __fmul_rn(d, d);
        if (dist < best_dist) {
            best_dist = dist;
            best = (uint32_t)j;
        }
    }
    return best;
}

// table[p] = nearest index of the 16-bit pattern p (fp16 or bf16).  Launch:
// 65536 threads in blocks of 256; dynamic shared memory n_c * 4 bytes.
__global__ void scalar_table(const float *__restrict__ centroids, int32_t n_c, bool bf16,
                             uint8_t *__restrict__ table)
{
    extern __shared__ float sc_tab[];
    for (int j = threadIdx.x; j < n_c; j += blockDim.x) sc_tab[j] = centroids[j];
    __syncthreads();
    const uint32_t p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p < 65536u) table[p] = (uint8_t)nearest(widen16((uint16_t)p, bf16), sc_tab, n_c);
}

// Eight 16-bit patterns -> their eight table bytes.
__device__ __forceinline__ uint2 lookup8(const uint8_t *tab, uint4 v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        lo |= (uint32_t)tab[w[k] & 0xffffu] << (16 * k);
        lo |= (uint32_t)tab[w[k] >> 16] << (16 * k + 8);
        hi |= (uint32_t)tab[w[k + 2] & 0xffffu] << (16 * k);
        hi |= (uint32_t)tab[w[k + 2] >> 16] << (16 * k + 8);
    }
    return make_uint2(lo, hi);
}

// out[e] = table[x[e]].  Launch: any grid of blocks of up to 1024 threads,
// dynamic shared memory 65536 bytes; grid-stride over 8-element units when
// `vec` (x 16-byte and out 8-byte aligned), the remaining elements one by one.
__global__ void __launch_bounds__(1024)
    scalar_lookup(const uint16_t *__restrict__ x, int64_t n, const uint8_t *__restrict__ table,
                  bool vec, uint8_t *__restrict__ out)
{
    extern __shared__ __align__(16) uint8_t sl_tab[];
    // the table must fit the launch's shared memory, else the block does
    // nothing (checked build; block-uniform); its lookups take 16-bit
    // patterns, so they stay inside it
    if (!vqk::dyn_smem_ok(sl_tab, 65536, 16)) return;
    const uint4 *t4 = reinterpret_cast<const uint4 *>(table);
    for (int k = threadIdx.x; k < 65536 / 16; k += blockDim.x)
        if (VQ_SPAN(t4 + k, 1, t4, 4096)) reinterpret_cast<uint4 *>(sl_tab)[k] = __ldg(t4 + k);
    __syncthreads();
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t units = vec ? n / 8 : 0;
    // four 16-byte loads in flight per thread before any lookup
    constexpr int U = 4;
    int64_t u = tid;
    for (; u + (U - 1) * nthreads < units; u += U * nthreads) {
        uint4 v[U];
#pragma unroll
        for (int k = 0; k < U; ++k)
            v[k] = VQ_VSPAN(x + (u + k * nthreads) * 8, 8, x, n, 16)
                       ? __ldcs(reinterpret_cast<const uint4 *>(x) + u + k * nthreads) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < U; ++k)
            if (VQ_VSPAN(out + (u + k * nthreads) * 8, 8, out, n, 8))
                __stcs(reinterpret_cast<uint2 *>(out) + u + k * nthreads, lookup8(sl_tab, v[k]));
    }
    for (; u < units; u += nthreads)
        if (VQ_VSPAN(x + u * 8, 8, x, n, 16) && VQ_VSPAN(out + u * 8, 8, out, n, 8))
            __stcs(reinterpret_cast<uint2 *>(out) + u,
                   lookup8(sl_tab, __ldcs(reinterpret_cast<const uint4 *>(x) + u)));
    for (int64_t e = units * 8 + tid; e < n; e += nthreads)
        if (VQ_SPAN(x + e, 1, x, n) && VQ_SPAN(out + e, 1, out, n)) out[e] = sl_tab[x[e]];
}

// ---- exact nearest centroid through the sorted codebook
//
// For a finite value y and finite centroids, let u_0 < ... < u_{m-1} be the
// distinct centroid values and rep[k] the lowest index j with c_j == u_k.
// D(u) = fl(fl(y - u)^2) is non-increasing in u up to y and non-decreasing
// after it (fl is monotone), so the distances equal to the least one form a
// run of consecutive u_k around y, and the rule's answer (lowest index among
// the least distances; none below +inf gives 0) is the least rep[k] over that
// run.  With L the last u_k <= y and R = L + 1, the least distance is
// min(D(u_L), D(u_R)); when the neighbours outside the pair are strictly
// larger, the run is {L}, {R} or {L, R}.  Anything else -- equal distances
// beyond the pair, or a non-finite value -- takes the scan of the rule itself.
struct SortedCb {
    const float *u;    // [m] distinct values, ascending
    const int *rep;    // [m] lowest original index of each value
    int m;
    int top;           // largest power of two <= m
};

// Build the sorted view in shared memory (all threads of the block; c[n_c]
// already in shared memory).  Returns false if a centroid is not finite (the
// scan is used for everything then).  u and rep need n_c entries, scratch
// (ints) n_c entries.
__device__ __forceinline__ bool build_sorted(const float *c, int n_c, float *u, int *rep,
                                             int *first, int *m_out)
{
    bool finite = true;
    for (int t = threadIdx.x; t < n_c; t += blockDim.x) {
        const float v = c[t];
        if (!(fabsf(v) <= 3.402823466e38f)) finite = false;
        int f = 1;
        for (int j = 0; j < t; ++j) f &= c[j] != v;  // the lowest index of its value
        first[t] = f;
    }
    finite = __syncthreads_and(finite) != 0;
    if (!finite) return false;
    for (int t = threadIdx.x; t < n_c; t += blockDim.x) {
        if (first[t]) {
            const float v = c[t];
            int rank = 0;
            for (int j = 0; j < n_c; ++j) rank += first[j] && c[j] < v;
            if (vqk::index_ok(rank, n_c)) {
                u[rank] = v;
                rep[rank] = t;
            }
        }
    }
    if (threadIdx.x == 0) {
        int m = 0;
        for (int j = 0; j < n_c; ++j) m += first[j];
        *m_out = m;
    }
    __syncthreads();
    return true;
}

__device__ __forceinline__ float dist_to(float y, float u)
{
    const float d = __fsub_rn(y, u);
    return __fmul_rn(d, d);
}

// Nearest index of y by the sorted view, or -1 if the scan must decide.
__device__ __forceinline__ int nearest_sorted(float y, const SortedCb &cb)
{
    if (!(fabsf(y) <= 3.402823466e38f)) return 0;  // NaN or inf: every distance NaN or inf
    int pos = 0;  // number of u_k <= y
    for (int step = cb.top; step > 0; step >>= 1)
        if (pos + step <= cb.m && cb.u[pos + step - 1] <= y) pos += step;
    const int L = pos - 1, R = pos;
    if (!vqk::index_ok(pos, cb.m + 1)) return -1;  // the scan decides (checked build)
    const float inf = __int_as_float(0x7f800000);
    const float dl = L >= 0 ? dist_to(y, cb.u[L]) : inf;
    const float dr = R < cb.m ? dist_to(y, cb.u[R]) : inf;
    const float best = fminf(dl, dr);
    if (best == inf) return 0;  // nothing below +inf
    const float dll = L >= 1 ? dist_to(y, cb.u[L - 1]) : inf;
    const float drr = R + 1 < cb.m ? dist_to(y, cb.u[R + 1]) : inf;
    const bool left = dl == best, right = dr == best;
    if ((left && !(dll > best)) || (right && !(drr > best))) return -1;  // a longer run
    if (left && right) return min(cb.rep[L], cb.rep[R]);
    return left ? cb.rep[L] : cb.rep[R];
}

// E consecutive elements of one row as fp32 (vector loads where E and the
// element size allow; rows are E-element aligned).
template <typename T, int E>
__device__ __forceinline__ void load_run(const T *p, float (&v)[E])
{
    constexpr int kBytes = E * (int)sizeof(T);
    if constexpr (kBytes >= 16 && kBytes % 16 == 0) {
        constexpr int kPer = 16 / (int)sizeof(T);
#pragma unroll
        for (int k = 0; k < E / kPer; ++k) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(p) + k);
            const T *t = reinterpret_cast<const T *>(&q);
#pragma unroll
            for (int i = 0; i < kPer; ++i) v[k * kPer + i] = widen_elem(t[i]);
        }
    } else if constexpr (kBytes == 8) {
        const uint2 q = __ldcs(reinterpret_cast<const uint2 *>(p));
        const T *t = reinterpret_cast<const T *>(&q);
#pragma unroll
        for (int i = 0; i < E; ++i) v[i] = widen_elem(t[i]);
    } else {
#pragma unroll
        for (int i = 0; i < E; ++i) v[i] = widen_elem(p[i]);
    }
}


// ---- exact nearest centroid of NC distinct centroids by cut points
//
// Let s_0 < ... < s_{NC-1} be the centroids sorted, orig(k) the original
// index of s_k, and d_j(v) = fl(fl(v - s_j)^2) the rule's distance.  On
// [s_k, s_{k+1}] d_k never decreases and d_{k+1} never increases as v grows,
// so "s_{k+1} beats s_k under the rule" (d_{k+1} < d_k, or d_{k+1} <= d_k when
// orig(k+1) < orig(k): ties go to the lower original index) is false at s_k,
// true at s_{k+1} and monotone in between.  Its first fp32 value t_k, found by
// a binary search over the bit patterns of that interval, is the cut point of
// the pair.  For lo <= v <= hi, k = #{j : t_j <= v} and the answer is
// orig(k): s_k beats or ties-and-wins against its two neighbours by the cut
// points, and every farther centroid is strictly farther than the
// neighbour between them, because the set-up only accepts codebooks whose
// neighbouring gaps differ by at most 2^15, whose gaps are at least 2^-40 and
// whose span [lo, hi] (the centroids widened by 2^15 outer gaps) stays below
// 2^62: a distance ratio of at least 1 + 2^-16 then survives the two
// roundings, with no underflow or overflow.  Values outside [lo, hi], NaN,
// and codebooks that fail those conditions take the rule's scan.
template <int NC>
struct CutCb {
    const float *t;   // [NC - 1] cut points, ascending, in shared memory
    float lo, hi;     // the values they decide
    uint64_t perm;    // orig(k) in bits 4k .. 4k + 3
    bool ok;          // the cut points apply (false: the scan for everything)
};

// Total order of the fp32 values as unsigned keys (finite values; -0 just
// below +0), and back.
__device__ __forceinline__ uint32_t f32_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float f32_from_key(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Block set-up (every thread of the block calls it; three block barriers).
// `sm` is shared memory for 4 NC floats; on return sm[NC .. 2 NC) holds the
// codebook as given, for the rule's scan.  Thread i < NC ranks centroid i;
// thread k < NC - 1 checks the gaps around pair (k, k + 1) and searches its
// cut point; every thread then reads the result.
template <int NC>
__device__ __forceinline__ void build_cut_cb(const float *__restrict__ centroids, float *sm,
                                             CutCb<NC> &cb)
{
    static_assert(NC >= 2 && NC <= 16, "4-bit original indices");
    float *srt = sm;                                      // [NC] ascending
    float *cgiven = sm + NC;                              // [NC] as given
    float *cut = sm + 2 * NC;                             // [NC - 1]
    int *orig = reinterpret_cast<int *>(sm + 3 * NC);     // [NC]
    const int t = threadIdx.x;
    bool ok = true;
    if (t < NC) {
        const float ci = __ldg(centroids + t);
        int rank = 0;
        bool distinct = true;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const float cj = __ldg(centroids + j);
            rank += cj < ci ? 1 : 0;
            distinct = distinct && (j >= t || cj != ci);
        }
        ok = fabsf(ci) <= 3.402823466e38f && distinct;
        cgiven[t] = ci;
        if (ok) {  // distinct finite values have distinct ranks 0 .. NC - 1
            srt[rank] = ci;
            orig[rank] = t;
        }
    }
    ok = __syncthreads_and(ok) != 0;
    bool pair_ok = true;
    if (ok && t < NC - 1) {
        const float a = srt[t], b = srt[t + 1];
        const float g = __fsub_rn(b, a);
        pair_ok = g >= 9.094947e-13f;  // 2^-40
        if (t + 1 < NC - 1) {          // neighbouring gaps within 2^15 of each other
            const float g2 = __fsub_rn(srt[t + 2], b);
            pair_ok = pair_ok && g2 <= 32768.f * g && g <= 32768.f * g2;
        }
        // the first fp32 value of [a, b] at which b beats a under the rule
        // (ties go to the lower original index)
        const bool upper_lower = orig[t + 1] < orig[t];
        uint32_t klo = f32_key(a), khi = f32_key(b);
        while (khi - klo > 1u) {  // at most 32 halvings
            const uint32_t km = klo + (khi - klo) / 2u;
            const float v = f32_from_key(km);
            const float da = __fmul_rn(__fsub_rn(v, a), __fsub_rn(v, a));
            const float db = __fmul_rn(__fsub_rn(v, b), __fsub_rn(v, b));
            const bool beats = upper_lower ? db <= da : db < da;
            if (beats) khi = km; else klo = km;
        }
        cut[t] = f32_from_key(khi);
    }
    ok = __syncthreads_and(ok && pair_ok) != 0;
    cb.ok = false;
    cb.lo = 0.f;
    cb.hi = 0.f;
    cb.perm = 0;
    cb.t = cut;
    if (ok) {
        const float lo = __fsub_rn(srt[0], __fmul_rn(32768.f, __fsub_rn(srt[1], srt[0])));
        const float hi = __fadd_rn(srt[NC - 1], __fmul_rn(32768.f, __fsub_rn(srt[NC - 1], srt[NC - 2])));
        cb.ok = __fsub_rn(hi, lo) <= 4.611686e18f;  // 2^62
        cb.lo = lo;
        cb.hi = hi;
#pragma unroll
        for (int k = 0; k < NC; ++k) cb.perm |= (uint64_t)(uint32_t)orig[k] << (4 * k);
    }
}

// Whether the cut points decide v (false for NaN, for values outside
// [lo, hi] and for codebooks that failed the set-up's conditions).
template <int NC>
__device__ __forceinline__ bool cut_decides(float v, const CutCb<NC> &cb)
{
    return cb.ok && v >= cb.lo && v <= cb.hi;
}

// The rule's answer for v through the cut points, valid when cut_decides(v):
// the original index of the k-th smallest centroid, k the number of cut
// points at or below v, by a branch-free binary search over the cut points
// in shared memory (the lanes read among NC - 1 consecutive words: no bank
// conflicts).  Callers take the rule's scan separately for the rare values
// the cut points do not decide.
template <int NC>
__device__ __forceinline__ int cut_rank(float v, const CutCb<NC> &cb)
{
    int k = 0;
#pragma unroll
    for (int step = NC / 2; step > 0; step >>= 1) k += v >= cb.t[k + step - 1] ? step : 0;
    return k;
}
template <int NC>
__device__ __forceinline__ uint32_t cut_code(float v, const CutCb<NC> &cb)
{
    return (uint32_t)(cb.perm >> (4 * cut_rank<NC>(v, cb))) & 15u;
}

// Randomised Hadamard rotation of rows of D = LPR * E elements, optionally
// fused with the scalar quantize.  LPR = lanes_per_row (a power of two up to
// 32, chosen by the host), 32 / LPR rows per warp; lane l of a row holds
// elements l*E .. l*E + E - 1.  Warps stride over groups of rows (a
// persistent grid), loading R groups before rotating the first.  The
// quantize of a codebook of exactly NC > 0 entries (2 to 16) counts the
// block's cut points (CutCb); with NC == 0 it searches the block's sorted
// view of the codebook (any size up to 256).  Launch: blockDim.x = 256,
// any grid; dynamic shared memory hadamard_smem(n_c) when QUANT and NC == 0,
// else 0.  x rows contiguous and E-element aligned (E * sizeof(T) up to 16
// bytes); idx 4-byte aligned when E % 4 == 0; y / idx [n_rows][D].
__host__ __device__ inline size_t hadamard_smem(int n_c) { return (size_t)n_c * 16 + 16; }

// The scalar quantize of any input type without a table: codebooks of 2, 4,
// 8 or 16 entries (NC) through the block's cut points, others (NC == 0)
// through the block's sorted view, every element falling back to the scan of
// the rule where they cannot decide.  A persistent grid strides over
// 8-element units (16-byte loads, two units in flight per thread, 8-byte
// stores) when `vec` (x 16-byte and out 8-byte aligned), then over the
// remaining elements one by one.  Launch: any grid of 256-thread blocks;
// dynamic shared memory hadamard_smem(n_c) when NC == 0, else 0.
template <typename T, int NC>
__global__ void __launch_bounds__(256)
    scalar_scan(const T *__restrict__ x, int64_t n, const float *__restrict__ centroids,
                int32_t n_c, bool vec, uint8_t *__restrict__ out);



template <typename T, int E, bool QUANT, int NC>
__global__ void __launch_bounds__(256)
    hadamard_rows(const T *__restrict__ x, const float *__restrict__ diag, int64_t n_rows,
                  int32_t lanes_per_row, float scale, const float *__restrict__ centroids,
                  int32_t n_c, float *__restrict__ y, uint8_t *__restrict__ idx)
{
    extern __shared__ float hq_sm[];
    SortedCb scb{nullptr, nullptr, 0, 0};
    const float *hq_cb = hq_sm;
    bool sorted_ok = false;
    // NC centroids (2 to 16): their cut points, set up once per block
    __shared__ float cut_sm[4 * 16];
    CutCb<(NC > 1 ? NC : 2)> cut;
    if constexpr (QUANT && NC > 0) {
        // the set-up reads NC <= n_c centroids (checked build: else the
        // block does nothing)
        if (!vqk::index_ok(NC - 1, n_c)) return;
        build_cut_cb<NC>(centroids, cut_sm, cut);
    }
    if constexpr (QUANT && NC == 0) {
        float *c = hq_sm;                                            // [n_c] as given
        float *u = c + n_c;                                          // [n_c] sorted distinct
        int *rep = reinterpret_cast<int *>(u + n_c);                 // [n_c]
        int *first = rep + n_c;                                      // [n_c]
        int *mcount = first + n_c;
        // the sorted view inside the launch's shared memory (checked build:
        // else the block does nothing; block-uniform)
        if (!vqk::dyn_smem_ok(hq_sm, hadamard_smem(n_c), 16)) return;
        for (int j = threadIdx.x; j < n_c; j += blockDim.x) c[j] = centroids[j];
        __syncthreads();
        sorted_ok = build_sorted(c, n_c, u, rep, first, mcount);
        if (sorted_ok) {
            scb.u = u;
            scb.rep = rep;
            scb.m = *mcount;
            int top = 1;
            while (top * 2 <= scb.m) top *= 2;
            scb.top = top;
        }
    }
    const int lane = threadIdx.x & 31;
    const int lpr = lanes_per_row;
    const int rows_per_warp = 32 / lpr;
    const int sub = lane / lpr;      // row within the warp
    const int l = lane - sub * lpr;  // lane within the row
    const int d = lpr * E;
    // R row groups per warp step, all loaded before any is rotated, so that
    // R loads per lane are in flight
    constexpr int R = E <= 4 ? 4 : E <= 16 ? 2 : 1;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    // the vector width of load_run
    constexpr uint32_t kRunBytes = E * sizeof(T);
    constexpr uint32_t kRunAlign = kRunBytes >= 16 && kRunBytes % 16 == 0 ? 16 : kRunBytes == 8 ? 8 : sizeof(T);
    // the row is lanes_per_row * E = d elements: diag and every row of x and
    // of the output hold d of them
    float dg[E];
#pragma unroll
    for (int j = 0; j < E; ++j) dg[j] = VQ_SPAN(diag + l * E + j, 1, diag, d) ? __ldg(diag + l * E + j) : 0.f;
    for (int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
         warp * R * rows_per_warp < n_rows; warp += warps) {  // warp-uniform
        float v[R][E];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = (warp * R + r) * rows_per_warp + sub;
            if (row < n_rows && VQ_VSPAN(x + (size_t)row * d + (size_t)l * E, E, x, n_rows * d, kRunAlign)) {
                load_run<T, E>(x + (size_t)row * d + (size_t)l * E, v[r]);
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) v[r][j] = 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = (warp * R + r) * rows_per_warp + sub;
            float *w = v[r];
#pragma unroll
            for (int j = 0; j < E; ++j) w[j] = __fmul_rn(w[j], dg[j]);
            // strides below E: pairs inside the lane's registers
#pragma unroll
            for (int s = 1; s < E; s <<= 1) {
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    if ((j & s) == 0) {
                        const float a = w[j], b = w[j + s];
                        w[j] = __fadd_rn(a, b);
                        w[j + s] = __fsub_rn(a, b);
                    }
                }
            }
            // strides E .. D/2: the partner element sits in lane l ^ (s / E)
            // (lower lane: own + partner; upper lane: partner - own, as
            // fma(-1, own, partner): the product is exact, so the one rounding
            // is that of the sum, bit for bit the add or subtract)
            for (int ls = 1; ls < lpr; ls <<= 1) {
                const float sg = (l & ls) != 0 ? -1.0f : 1.0f;
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const float q = __shfl_xor_sync(0xffffffffu, w[j], ls);
                    w[j] = __fmaf_rn(sg, w[j], q);
                }
            }
            if (row >= n_rows) continue;
#pragma unroll
            for (int j = 0; j < E; ++j) w[j] = __fmul_rn(w[j], scale);
            if constexpr (QUANT) {
                uint32_t code[E];
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    if constexpr (NC > 0) {
                        code[j] = cut_code<NC>(w[j], cut);
                    } else {
                        const int k = sorted_ok ? nearest_sorted(w[j], scb) : -1;
                        code[j] = k >= 0 ? (uint32_t)k : nearest(w[j], hq_cb, n_c);
                    }
                }
                if constexpr (NC > 0) {
                    // values the cut points do not decide (rare): the rule's scan
                    bool all = true;
#pragma unroll
                    for (int j = 0; j < E; ++j) all = all && cut_decides<NC>(w[j], cut);
                    if (!all) {
#pragma unroll
                        for (int j = 0; j < E; ++j)
                            if (!cut_decides<NC>(w[j], cut)) code[j] = nearest(w[j], cut_sm + NC, NC);
                    }
                }
                uint8_t *o = idx + (size_t)row * d + (size_t)l * E;
                if (!VQ_VSPAN(o, E, idx, n_rows * d, E % 4 == 0 ? 4 : 1)) continue;
                if constexpr (E % 4 == 0) {
#pragma unroll
                    for (int j = 0; j < E; j += 4)
                        *reinterpret_cast<uint32_t *>(o + j) =
                            code[j] | code[j + 1] << 8 | code[j + 2] << 16 | code[j + 3] << 24;
                } else {
#pragma unroll
                    for (int j = 0; j < E; ++j) o[j] = (uint8_t)code[j];
                }
            } else {
                float *o = y + (size_t)row * d + (size_t)l * E;
                if (!VQ_SPAN(o, E, y, n_rows * d)) continue;
#pragma unroll
                for (int j = 0; j < E; ++j) o[j] = w[j];
            }
        }
    }
}

}  // namespace vqs

namespace vqs {

// out[e] = centroids[idx[e]] converted to the output type (round to
// nearest); an index >= n_c gives 0.  Launch: any grid, grid-stride.
template <typename T>
__global__ void __launch_bounds__(256)
    scalar_dequant(const uint8_t *__restrict__ idx, int64_t n, const float *__restrict__ centroids,
                   int32_t n_c, T *__restrict__ out)
{
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += nthreads) {
        const uint32_t k = idx[e];
        const float v = k < (uint32_t)n_c ? __ldg(centroids + k) : 0.f;
        if constexpr (sizeof(T) == 4) {
            out[e] = v;
        } else if constexpr (std::is_same<T, __half>::value) {
            out[e] = __float2half_rn(v);
        } else {
            out[e] = __float2bfloat16_rn(v);
        }
    }
}

// Eight consecutive elements (16-byte aligned) as fp32.
template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&v)[8])
{
    if constexpr (sizeof(T) == 4) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
        v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
    } else {
        const uint4 q = __ldcs(reinterpret_cast<const uint4 *>(p));
        const T *t = reinterpret_cast<const T *>(&q);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = widen_elem(t[i]);
    }
}

template <typename T, int NC>
__global__ void __launch_bounds__(256)
    scalar_scan(const T *__restrict__ x, int64_t n, const float *__restrict__ centroids,
                int32_t n_c, bool vec, uint8_t *__restrict__ out)
{
    extern __shared__ float ss_sm[];
    SortedCb scb{nullptr, nullptr, 0, 0};
    bool sorted_ok = false;
    __shared__ float cut_sm[4 * 16];
    CutCb<(NC > 1 ? NC : 2)> cut;
    if constexpr (NC > 0) {
        build_cut_cb<NC>(centroids, cut_sm, cut);
    } else {
        float *c = ss_sm;
        float *u = c + n_c;
        int *rep = reinterpret_cast<int *>(u + n_c);
        int *first = rep + n_c;
        int *mcount = first + n_c;
        for (int j = threadIdx.x; j < n_c; j += blockDim.x) c[j] = centroids[j];
        __syncthreads();
        sorted_ok = build_sorted(c, n_c, u, rep, first, mcount);
        if (sorted_ok) {
            scb.u = u;
            scb.rep = rep;
            scb.m = *mcount;
            int top = 1;
            while (top * 2 <= scb.m) top *= 2;
            scb.top = top;
        }
    }
    auto quant = [&](float v) -> uint32_t {
        if constexpr (NC > 0) {
            return cut_decides<NC>(v, cut) ? cut_code<NC>(v, cut) : nearest(v, cut_sm + NC, NC);
        } else {
            const int k = sorted_ok ? nearest_sorted(v, scb) : -1;
            return k >= 0 ? (uint32_t)k : nearest(v, ss_sm, n_c);
        }
    };
    auto quant8 = [&](const float (&v)[8]) -> uint2 {
        uint32_t lo = 0, hi = 0;
        if constexpr (NC > 0) {
            // branch-free for the values the cut points decide; the rule's
            // scan (rare) only when one of the eight is not
            bool all = true;
#pragma unroll
            for (int i = 0; i < 8; ++i) all = all && cut_decides<NC>(v[i], cut);
            if (all) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    lo |= cut_code<NC>(v[i], cut) << (8 * i);
                    hi |= cut_code<NC>(v[i + 4], cut) << (8 * i);
                }
                return make_uint2(lo, hi);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo |= quant(v[i]) << (8 * i);
            hi |= quant(v[i + 4]) << (8 * i);
        }
        return make_uint2(lo, hi);
    };
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    // 8-element units (x 16-byte and out 8-byte aligned when `vec`), two
    // units' loads in flight per thread; then the remaining elements
    const int64_t units = vec ? n / 8 : 0;
    constexpr int U = 2;
    int64_t u = tid;
    for (; u + (U - 1) * nthreads < units; u += U * nthreads) {
        float v[U][8];
#pragma unroll
        for (int k = 0; k < U; ++k) load8<T>(x + (u + k * nthreads) * 8, v[k]);
#pragma unroll
        for (int k = 0; k < U; ++k) __stcs(reinterpret_cast<uint2 *>(out) + u + k * nthreads, quant8(v[k]));
    }
    for (; u < units; u += nthreads) {
        float v[8];
        load8<T>(x + u * 8, v);
        __stcs(reinterpret_cast<uint2 *>(out) + u, quant8(v));
    }
    for (int64_t e = units * 8 + tid; e < n; e += nthreads) out[e] = (uint8_t)quant(widen_elem(x[e]));
}

// ---- fp16 keys against 2, 4, 8 or 16 centroids: a bucket table from the cut points
//
// An fp16 pattern h falls in bucket h >> 6 (sign, exponent and the top four
// significand bits: 1,024 buckets); over a bucket the value moves
// monotonically with h & 63 (up in positive buckets, down in negative ones).
// Where the cut points decide both end values of a bucket they decide all of
// it, and the rank (cut points at or below the value) is monotone over it.
// So a bucket whose end ranks differ by at most one has at most one change
// of code: its entry holds the code below the change (A), the code from it
// on (B) and the first pattern T that takes B.  The other buckets (two or
// more changes; the values the cut points leave to the scan: NaN,
// infinities, keys outside [lo, hi]; every bucket when the codebook fails
// the cut points' conditions) are flagged, and their elements take cut_code
// or the rule's scan one by one.  The result is the cut points' (or the
// scan's) answer for every pattern, bit for bit.
//
// Entry (32 bits): T in bits 16-31, A in bits 0-3, B in bits 8-11, the flag
// in bits 7 and 15 (T = 0 when flagged or when the bucket has one code).  With
// hx = h << 16 | 0xffff, h < T exactly when hx < entry, so the code byte is
// the low byte of entry (A) or of entry >> 8 (B), the flag in its bit 7.
// The 1,024 entries (4 KiB) are copied once per shared-memory bank: lane l
// finds bucket b at byte (b * 32 + l) * 4, in its own bank whatever b is, so
// a warp's 32 lookups take one wavefront (random bytes of a 64 KiB table
// take about four).
constexpr uint32_t kBucketFlag = 0x8080u;
constexpr int kBucketCopyBytes = 131072;  // 1,024 entries x 32 banks x 4 bytes
constexpr int kBucketSmemBytes = kBucketCopyBytes + 4096;

template <int NC>
__device__ uint32_t bucket_entry(uint32_t b, const CutCb<NC> &cb)
{
    const uint32_t base = b << 6;
    const float v0 = widen16((uint16_t)base, false);
    const float v1 = widen16((uint16_t)(base | 63u), false);
    if (!cut_decides<NC>(v0, cb) || !cut_decides<NC>(v1, cb)) return kBucketFlag;
    const int k0 = cut_rank<NC>(v0, cb), k1 = cut_rank<NC>(v1, cb);
    const uint32_t c0 = (uint32_t)(cb.perm >> (4 * k0)) & 15u;
    const uint32_t c1 = (uint32_t)(cb.perm >> (4 * k1)) & 15u;
    if (k0 == k1) return c0 | c0 << 8;
    if (k1 - k0 != 1 && k0 - k1 != 1) return kBucketFlag;
    // rank(lo) == k0, rank(hi) == k1: the first position of rank k1
    uint32_t lo = 0, hi = 63;
    while (hi - lo > 1u) {
        const uint32_t mid = (lo + hi) / 2u;
        if (cut_rank<NC>(widen16((uint16_t)(base | mid), false), cb) == k1) hi = mid; else lo = mid;
    }
    return (base | hi) << 16 | c0 | c1 << 8;
}

// The code byte (flag in bit 7) of pattern h from its entry; hx = h << 16 | 0xffff.
__device__ __forceinline__ uint32_t bucket_byte(uint32_t e, uint32_t hx)
{
    return hx < e ? e : e >> 8;
}

// out[e] = the rule's index of fp16 x[e] for a codebook of exactly NC
// entries.  Launch: any grid of blocks of up to 1024 threads (one block per
// SM builds the table once), dynamic shared memory kBucketSmemBytes;
// grid-stride over 8-element units when `vec` (x 16-byte and out 8-byte
// aligned), the remaining elements one by one.
template <int NC>
__global__ void __launch_bounds__(1024)
    scalar_bucket(const uint16_t *__restrict__ x, int64_t n, const float *__restrict__ centroids,
                  bool vec, uint8_t *__restrict__ out)
{
    extern __shared__ __align__(16) uint8_t sb_tab[];
    __shared__ float cut_sm[4 * 16];
    // the copies and the entries must fit the launch's shared memory, else the
    // block does nothing (checked build; block-uniform); the lookups' offsets
    // stay below kBucketCopyBytes by construction
    if (!vqk::dyn_smem_ok(sb_tab, kBucketSmemBytes, 16)) return;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t units = vec ? n / 8 : 0;
    auto load = [&](int64_t k) -> uint4 {
        return VQ_VSPAN(x + k * 8, 8, x, n, 16) ? __ldcs(reinterpret_cast<const uint4 *>(x) + k)
                                                : make_uint4(0, 0, 0, 0);
    };
    // U units per thread and step; the next step's loads are issued before
    // the current step's lookups, and the first step's before the set-up
    constexpr int U = 2;
    int64_t u = tid;
    uint4 cur[U];
    const bool first = u + (U - 1) * nthreads < units;
    if (first) {
#pragma unroll
        for (int k = 0; k < U; ++k) cur[k] = load(u + k * nthreads);
    }
    // the block's units of the next kPrefetchSteps steps (blockDim.x
    // consecutive units per step and k) are brought into L2 during the set-up
    constexpr int kPrefetchSteps = 3;
    if (threadIdx.x == 0) {
        const int64_t b0 = (int64_t)blockIdx.x * blockDim.x;
        for (int st = 1; st <= kPrefetchSteps; ++st)
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int64_t a = b0 + (int64_t)(st * U + k) * nthreads;
                const int64_t c = units - a < (int64_t)blockDim.x ? units - a : (int64_t)blockDim.x;
                if (c > 0 && VQ_VSPAN(x + a * 8, c * 8, x, n, 16))
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                                 :: "l"(x + a * 8), "r"((uint32_t)(c * 16)) : "memory");
            }
    }
    CutCb<NC> cb;
    build_cut_cb<NC>(centroids, cut_sm, cb);
    uint32_t *entries = reinterpret_cast<uint32_t *>(sb_tab + kBucketCopyBytes);
    for (uint32_t b = threadIdx.x; b < 1024u; b += blockDim.x)
        entries[b] = cb.ok ? bucket_entry<NC>(b, cb) : kBucketFlag;
    __syncthreads();
    {
        uint32_t *copies = reinterpret_cast<uint32_t *>(sb_tab);
        for (int i = threadIdx.x; i < kBucketCopyBytes / 4; i += blockDim.x) copies[i] = entries[i >> 5];
    }
    __syncthreads();
    const uint8_t *mine = sb_tab + (threadIdx.x & 31u) * 4u;
    // entry of the pattern in bits 0-15 (lo) or 16-31 (hi) of w
    auto entry_lo = [&](uint32_t w) -> uint32_t {
        return *reinterpret_cast<const uint32_t *>(mine + ((w & 0xffc0u) << 1));
    };
    auto entry_hi = [&](uint32_t w) -> uint32_t {
        return *reinterpret_cast<const uint32_t *>(mine + ((w >> 15) & 0x1ff80u));
    };
    auto slow = [&](uint32_t h) -> uint32_t {
        const float v = widen16((uint16_t)h, false);
        return cut_decides<NC>(v, cb) ? cut_code<NC>(v, cb) : nearest(v, cut_sm + NC, NC);
    };
    // four patterns (two words) -> four code bytes
    auto quant4 = [&](uint32_t w0, uint32_t w1) -> uint32_t {
        const uint32_t b0 = bucket_byte(entry_lo(w0), __byte_perm(w0, 0xffffffffu, 0x1044));
        const uint32_t b1 = bucket_byte(entry_hi(w0), w0 | 0xffffu);
        const uint32_t b2 = bucket_byte(entry_lo(w1), __byte_perm(w1, 0xffffffffu, 0x1044));
        const uint32_t b3 = bucket_byte(entry_hi(w1), w1 | 0xffffu);
        uint32_t r = __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
        if (r & 0x80808080u) {  // rare: the flagged elements one by one
            const uint32_t h[4] = {w0 & 0xffffu, w0 >> 16, w1 & 0xffffu, w1 >> 16};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if ((r >> (8 * i)) & 0x80u) r = (r & ~(0xffu << (8 * i))) | slow(h[i]) << (8 * i);
        }
        return r;
    };
    auto quant8 = [&](uint4 q) -> uint2 { return make_uint2(quant4(q.x, q.y), quant4(q.z, q.w)); };
    auto store = [&](int64_t k, uint2 r) {
        if (VQ_VSPAN(out + k * 8, 8, out, n, 8)) __stcs(reinterpret_cast<uint2 *>(out) + k, r);
    };
    if (first) {
        for (;;) {
            const int64_t nu = u + U * nthreads;
            const bool more = nu + (U - 1) * nthreads < units;
            uint4 nxt[U];
            if (more) {
#pragma unroll
                for (int k = 0; k < U; ++k) nxt[k] = load(nu + k * nthreads);
            }
#pragma unroll
            for (int k = 0; k < U; ++k) store(u + k * nthreads, quant8(cur[k]));
            u = nu;
            if (!more) break;
#pragma unroll
            for (int k = 0; k < U; ++k) cur[k] = nxt[k];
        }
    }
    for (; u < units; u += nthreads) store(u, quant8(load(u)));
    for (int64_t e = units * 8 + tid; e < n; e += nthreads)
        if (VQ_SPAN(x + e, 1, x, n) && VQ_SPAN(out + e, 1, out, n)) {
            const uint32_t h = x[e];
            const uint32_t byte = bucket_byte(entry_lo(h), h << 16 | 0xffffu) & 0xffu;
            out[e] = (uint8_t)((byte & 0x80u) ? slow(h) : byte);
        }
}

}  // namespace vqs
