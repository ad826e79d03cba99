// vq_tc.cuh -- exact product-VQ encode with the screening contraction on the
// 5th-generation tensor cores (tcgen05, accumulator in tensor memory).
//
// Same scheme and the same proof as vq_filter.cuh, with one change: the
// screening values s~(c) = |c|^2 - 2 x.c of a tile of 128 rows against all
// centroids come from one tcgen05.mma of kind::tf32 per 256 centroids,
//     A (128 x K, rows)      = [x_0 .. x_SUB-1, 1, 1, 1, 0 ...]
//     B (n_pad x K, centroids) = [-2c_0 .. -2c_SUB-1, n_hi, n_mid, n_lo, 0 ...]
// where n_hi + n_mid + n_lo is the fp32 |c|^2 split into three tf32 pieces.
// fp16 and bf16 values, -2c and 1 are exact in tf32, so every product is
// exact; only the accumulation inside the tensor core rounds.  Its error is
// bounded by eps_tc times the sum of the magnitudes of the terms, which is at
// most 2 (C2 + sum_i |x_i| A_i).  eps_tc = 2^-16 is taken: 8 times the error
// of an fp32 accumulator that truncates each of K = 16 partial sums, and 25
// times the largest error that tests/test_tc_accumulation.py measures on
// GB300 through this file's own MMA, descriptors and tensor-memory loads
// (2^-20.7, chains of up to 6 MMAs, on cancelling, many-decade, split-piece,
// near-underflow and screening-operand score sets).  Adding the
// rounding of the fp32 |c|^2 (gamma_SUB) gives the screening bound
//     B(x) = (2 eps_tc + 2 gamma_SUB) (C2 + sum_i |x_i| A_i),
// and the threshold, candidate groups, exact re-evaluation and exact queue
// follow as in vq_filter.cuh.
//
// fp32 rows and codebooks are not exact in tf32.  The rows are split as
// below (x = hi + mid + lo), and -2c likewise into b_hi + b_mid + b_lo with
// a second B piece holding b_mid; three accumulating MMAs form (hi, b_hi),
// (mid, b_hi) and (hi, b_mid).  The dropped products x_lo (-2c), x b_lo and
// mid b_mid are each at most 2^-20 |x| |2c|, together 3 x 2^-19 sum_i |x_i|
// A_i (the kernel adds 2^-17) to the screening bound.
//
// With SMOOTH, each row is first divided by its per-channel smooth factors
// (fp32, rounded to nearest), and the divided row -- an fp32 value, not
// exact in tf32 -- is what is encoded.  Each element is x_i = hi_i + mid_i +
// lo_i exactly (hi keeps the top 11 significant bits, mid the next 11 of the
// exact remainder, lo the last 2, |lo_i| <= 2^-20 |x_i|).  Two accumulating
// MMAs multiply A_hi = [hi, 1, 1, 1, 0 ...] and A_mid = [mid, 0 ...] by the
// same B, so every product is exact; the dropped lo part changes the score
// by |2 sum_i lo_i c_i| <= 2^-19 sum_i |x_i| A_i.  The magnitudes of the
// terms add up to at most (1 + 2^-9) times their bound above, and the kernel
// uses B(x) = (2 (1 + 2^-9) eps_tc + 2 gamma_SUB + 2^-19) (C2 + sum_i |x_i|
// A_i); the accumulation spans 2 K terms, 16 or 32, whose truncating fp32
// error (at most 32 x 2^-23 = 2^-18 of the magnitudes) eps_tc still covers.
//
// Underflow.  The relative bounds above hold for normal numbers.  Below
// 2^-126 a split drops up to 2^-136 absolute (the mask keeps no bit of a
// subnormal below 2^-136), and the tensor core may flush subnormal operands,
// products or partial sums.  A flushed or dropped part of x (below 2^-126 per
// element) costs at most 2^-125 A_i per term, which 2^-100 covers while
// A_i <= 2^22 and 2^-15 C2 (C2 >= A_i^2 up to rounding) covers beyond.  A
// flushed or dropped part of -2c (below 2^-125) costs at most 2^-125 |x_i|,
// which the A_i term covers once A_i is floored at 2^-100 (2^-15 x 2^-100 =
// 2^-115); a larger bound only widens the candidate set.  Rounding the
// |c|^2 pieces drops below 2^-136.  Each of these is a few 2^-125 terms
// next to the 2^-100 that bnd and thr carry.
//
// The accumulator of a tile is a 128-lane x n_pad-column fp32 block of tensor
// memory, so thread t of the block owns row t of the tile: it reads its own
// row's scores (tcgen05.ld) and reduces them without any exchange.
//
// Every thread waits for each pass's MMA on the mbarrier, polling at most
// kWaitPolls times; a wait that needed more than POLLS polls, or never
// completed, counts as given up (in the library POLLS is kWaitPolls, so only
// the latter; smaller values exist only to test this path).  The block
// agrees once per tile, after the tile's passes, on whether any wait gave up.
// A wait that completed late still completed before the thread reads the
// scores, so no tensor-memory load races an MMA unless a wait never
// completed.  The waits use the barrier's phase parity, which only tells the
// last two phases apart, so at most one phase is ever outstanding: thread 0
// starts a pass's phase only after its own wait for the previous one; once a
// wait of its own has given up it issues no more MMAs and completes each
// later pass's phase with a plain arrive instead (so every pass still
// completes one phase), and once a wait of its own never completed it starts
// no phase at all.  If a wait gave up, thread 0 waits (kWaitPolls) for the
// last phase it started, the block marks every row it has not encoded with
// 0xFFFFFFFF, sets kStatusWaitGaveUp in the device status word and frees the
// tensor memory: never while an MMA it issued is in flight, unless a wait
// never completed.
//
// Launch: block = 128 * TPS threads; dynamic shared memory =
// TcLayout::bytes(...) (at least 512/(NCOL * TPS) CTAs' worth of a 228 KiB SM,
// which caps the CTAs per SM at the tensor-memory budget: NCOL * TPS columns
// each); grid.x = n_groups * blocks_per_group, each block encoding
// tiles_per_block consecutive 128-row tiles of one group, TPS at a time (a
// step): thread t works on tile t / 128 of the step, row t % 128, and the
// step's tiles share each pass's commit, wait and barrier.  Requirements: T is __half, __nv_bfloat16 or float, 64 <= n_centroids <=
// 256, x aligned to SUB * sizeof(T) bytes.  With SMOOTH: `smooth`
// [n_groups][smooth_ns * SUB] fp32 factors, row m of a group holding channels
// (m % smooth_ns) * SUB + i; TcLayout's A holds two pieces (NA = 2).
#pragma once

#include <type_traits>

#include "vq_check.cuh"
#include "vq_filter.cuh"
#include "vq_kernels.cuh"
#include "vq_status.cuh"
#include "vq_umma.cuh"

namespace vqk {

#ifdef VQ_TC_STATS
// Test builds only: rows per screening outcome, [cnt 1, cnt 1 tight, cnt 2,
// cnt 2 tight, queued]; "tight" = the least excluded group minimum lies
// within one bound of the threshold.
static __device__ unsigned long long g_tc_stats[8];
#endif

// Least of N values by a tree of three-input minima (NaN ignored unless all
// are NaN, as min3).  W is float, or uint32_t holding float bits.
template <int N, typename W>
__device__ __forceinline__ float tree_min_p(const W *w)
{
    auto f = [](W v) -> float {
        if constexpr (std::is_same<W, float>::value) return v;
        else return __uint_as_float(v);
    };
    if constexpr (N == 1) {
        return f(w[0]);
    } else if constexpr (N == 2) {
        return fminf(f(w[0]), f(w[1]));
    } else if constexpr (N == 3) {
        return min3(f(w[0]), f(w[1]), f(w[2]));
    } else {
        constexpr int a = (N + 2) / 3, b = (N - a + 1) / 2, c = N - a - b;
        return min3(tree_min_p<a>(w), tree_min_p<b>(w + a), tree_min_p<c>(w + a + b));
    }
}

// Least of GC consecutive scores (float bits) by a shallow tree of
// three-input minima: 8 operations in 3 levels for 16, 4 in 2 for 8.
template <int GC>
__device__ __forceinline__ float group_min(const uint32_t *u)
{
    auto f = [&](int i) { return __uint_as_float(u[i]); };
    if constexpr (GC == 16) {
        const float a = min3(min3(f(0), f(1), f(2)), min3(f(3), f(4), f(5)), min3(f(6), f(7), f(8)));
        const float b = min3(min3(f(9), f(10), f(11)), min3(f(12), f(13), f(14)), f(15));
        return fminf(a, b);
    } else {
        return tree_min_p<GC>(u);
    }
}
template <int N>
__device__ __forceinline__ float tree_min(const float (&w)[N])
{
    return tree_min_p<N>(&w[0]);
}

// Keep the top 10 bits of an fp32 significand (the tf32 value, exactly).
__device__ __forceinline__ float tf32_trunc(float v) { return __uint_as_float(__float_as_uint(v) & 0xffffe000u); }

// ------------------------------------------------------------------ layout

template <int SUB, int NCOL, int GC, int NA = 1, int NB = 1, int TPS = 1>
struct TcLayout {
    static constexpr int kK = SUB == 4 ? 8 : 16;       // MMA K (tf32 elements), 8 per instruction
    static constexpr int kRowBytes = kK * 4;
    static constexpr int kGC = GC;                       // centroids per screening group
    // exact layout: per group, centroid pairs interleaved -- component i of
    // centroids (2p, 2p+1) is the float2 (-c_2p_i, -c_2p+1_i) -- so one packed
    // f32x2 evaluation covers two centroids; one 16-byte pad per group
    static constexpr int kGroupFloats = kGC * SUB + 4;
    static constexpr int kCtasPerSm = 512 / (NCOL * TPS);
    __host__ __device__ static int padded(int nc) { return (nc + 31) / 32 * 32; }
    __host__ __device__ static int groups(int nc) { return padded(nc) / kGC; }
    // byte offsets
    static constexpr size_t kABytes = (size_t)128 * kRowBytes;  // one A piece of one tile
    __host__ __device__ static size_t a_off() { return 0; }  // tile h of a step: its NA pieces at h * NA * kABytes
    __host__ __device__ static size_t b_off() { return TPS * NA * kABytes; }
    __host__ __device__ static size_t x_off(int /*nc: B always holds 256 rows*/) { return b_off() + (size_t)NB * 256 * kRowBytes; }
    __host__ __device__ static size_t misc_off(int nc)
    {
        return x_off(nc) + (size_t)groups(nc) * kGroupFloats * 4;
    }
    // misc: SUB + 1 maxima, queue counter, tensor-memory address, pad, mbarrier (8-aligned), queue
    __host__ __device__ static size_t used(int nc) { return misc_off(nc) + 64 + 128 * TPS * 4; }
    __host__ __device__ static size_t bytes(int nc)
    {
        const size_t cap = (size_t)228 * 1024 / (kCtasPerSm + 1) + 1024;
        const size_t u = used(nc) + 1024;  // room to align the base to 1 KiB
        return u > cap ? u : cap;
    }
};

// Per sub_dim, and per whether each row is carried as two tf32 pieces
// (SPLIT: smoothed rows or fp32 keys): tensor-memory columns per tile,
// centroids per screening group, minimum CTAs per SM (register budget), tiles
// per step (a CTA has 128 threads per tile of a step and screens the step's
// tiles with one commit, one wait and one barrier per pass).  Measured best on
// GB300 for 256-centroid codebooks; two tiles per step pay only for 16-bit
// rows at sub_dim 4, where the per-pass synchronisation is the larger share.
template <int SUB, bool SPLIT = false>
struct TcConfig;
template <>
struct TcConfig<4, false> {
    static constexpr int kCols = 64, kGroup = 16, kMinBlocks = 4, kTps = 2;
};
template <>
struct TcConfig<4, true> {
    static constexpr int kCols = 64, kGroup = 16, kMinBlocks = 8, kTps = 1;
};
template <>
struct TcConfig<8, false> {
    static constexpr int kCols = 64, kGroup = 8, kMinBlocks = 6, kTps = 1;
};
template <>
struct TcConfig<8, true> : TcConfig<8, false> {};

// ------------------------------------------------------------------ kernel

template <typename T, int SUB, int NCOL, int GC, int MINB, typename OutT = uint32_t,
          bool SMOOTH = false, int POLLS = kWaitPolls, int TPS = 1>
__global__ void __launch_bounds__(128 * TPS, MINB)
    encode_tc(const T *__restrict__ x, const T *__restrict__ codebooks, int64_t n_per_group,
              int32_t n_centroids, int64_t blocks_per_group, int32_t tiles_per_block, float one,
              OutT *__restrict__ out, const float *__restrict__ smooth, int32_t smooth_ns)
{
    static_assert(SUB == 4 || SUB == 8, "sub_dim 4 or 8");
    static_assert(NCOL == 32 || NCOL == 64 || NCOL == 128 || NCOL == 256, "tensor-memory columns");
    static_assert(GC == 8 || GC == 16, "centroid group size");
    constexpr bool kF32 = std::is_same<T, float>::value;  // fp32 rows and codebook
    constexpr int kNA = SMOOTH || kF32 ? 2 : 1;  // A pieces: rows not exact in tf32
    constexpr int kNB = kF32 ? 2 : 1;            // B pieces: -2c not exact in tf32
    using L = TcLayout<SUB, NCOL, GC, kNA, kNB, TPS>;
    constexpr int THREADS = 128 * TPS;
    constexpr int kK = L::kK;
    constexpr int kKB = kK / 4;  // 16-byte core-matrix columns per row
    constexpr int kGC = L::kGC;
    constexpr int kNG = 256 / kGC;  // most groups a codebook can have
    constexpr uint32_t kQueued = 0xffffffffu;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *sa = reinterpret_cast<float *>(sm + L::a_off());
    float *sb = reinterpret_cast<float *>(sm + L::b_off());
    float *sx = reinterpret_cast<float *>(sm + L::x_off(n_centroids));
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::misc_off(n_centroids));
    uint32_t *smax = misc;              // [0] = C2, [1 + i] = A_i
    uint32_t *qcount = misc + SUB + 1;
    uint32_t *tslot = misc + SUB + 2;
    uint64_t *bar = reinterpret_cast<uint64_t *>(misc + 12);  // 48 bytes in: 8-aligned
    uint32_t *queue = misc + 16;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int th = tid >> 7;   // tile of the step this thread works on
    const int rt = tid & 127;  // its row in that tile, its tensor-memory lane
    const int n_pad = L::padded(n_centroids);
    const int64_t g = blockIdx.x / blocks_per_group;
    const int64_t blk = blockIdx.x - g * blocks_per_group;
    const T *__restrict__ cb = codebooks + (size_t)g * (size_t)n_centroids * SUB;
    const T *__restrict__ xg = x + (size_t)g * (size_t)n_per_group * SUB;
    OutT *__restrict__ og = out + (size_t)g * (size_t)n_per_group;
    const float *__restrict__ sg = SMOOTH ? smooth + (size_t)g * (size_t)smooth_ns * SUB : nullptr;
    const int64_t row_base = blk * (int64_t)tiles_per_block * 128;

    // buffer extents, for the checked build's bounds checks (vq_check.cuh)
    const int64_t n_groups_all = gridDim.x / blocks_per_group;
    const int64_t nx = n_groups_all * n_per_group * SUB, nout = n_groups_all * n_per_group;
    constexpr uint64_t kSaBytes = TPS * kNA * L::kABytes, kSbBytes = (uint64_t)kNB * 256 * L::kRowBytes;
    const uint64_t sx_bytes = (uint64_t)L::groups(n_centroids) * L::kGroupFloats * 4;
    constexpr uint64_t kMiscBytes = 64 + 128 * TPS * 4;
    constexpr uint32_t kRowAlign = SUB * sizeof(T) < 16 ? SUB * sizeof(T) : 16;  // load_row
    if constexpr (kChecked) {
        // the layout inside the launch's shared memory, the block inside the
        // grid, its smooth factors inside theirs: else the block does nothing
        if (!dyn_smem_ok(sm, L::used(n_centroids), 16) || !span_ok(bar, 8, misc, kMiscBytes, 8) ||
            !span_ok(queue, 512 * TPS, misc, kMiscBytes, 4) || !index_ok(g, n_groups_all) ||
            (SMOOTH && !VQ_SPAN(sg, (int64_t)smooth_ns * SUB, smooth, n_groups_all * smooth_ns * SUB)))
            return;  // block-uniform
    }

    // ---- set-up: maxima, barrier, tensor memory, constant part of A
    if (tid < SUB + 2) misc[tid] = 0u;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tslot)),
                     "r"(NCOL * TPS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    {
        // A row rt of tile th: columns SUB.. of the row are the constant
        // [1, 1, 1, 0 ...] in the first piece and zero in the others
#pragma unroll
        for (int pc = 0; pc < kNA; ++pc) {
            float *arow = sa + (th * kNA + pc) * (L::kABytes / 4);
#pragma unroll
            for (int kb = SUB / 4; kb < kKB; ++kb) {
                const float4 v = kb == SUB / 4 && pc == 0 ? make_float4(1.f, 1.f, 1.f, 0.f)
                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                float4 *dst = reinterpret_cast<float4 *>(arow + ((rt >> 3) * (kKB * 128) + kb * 128 + (rt & 7) * 16) / 4);
                if (span_ok(dst, 16, sa, kSaBytes, 16)) *dst = v;
            }
        }
    }
    __syncthreads();

    // ---- stage the codebook: B operand, exact layout, maxima
    for (int c = tid; c < 256; c += THREADS) {
        const bool real = c < n_centroids;
        const bool cb_ok = !real || VQ_SPAN(cb + (size_t)c * SUB, SUB, codebooks, n_groups_all * n_centroids * SUB);
        float v[SUB];
#pragma unroll
        for (int i = 0; i < SUB; ++i) v[i] = real && cb_ok ? widen(cb[(size_t)c * SUB + i]) : 0.f;
        float nrm = mul_rn(v[0], v[0]);
#pragma unroll
        for (int i = 1; i < SUB; ++i) nrm = fma_rn(v[i], v[i], nrm);
        float bk[kK];
#pragma unroll
        for (int k = 0; k < kK; ++k) bk[k] = 0.f;
        float bm[SUB];  // second piece of -2c (fp32 codebooks)
#pragma unroll
        for (int i = 0; i < SUB; ++i) {
            const float w = -2.0f * v[i];
            bk[i] = kF32 ? tf32_trunc(w) : w;
            bm[i] = kF32 ? tf32_trunc(w - bk[i]) : 0.f;
        }
        if (real) {
            const float hi = tf32_trunc(nrm);
            const float mid = tf32_trunc(nrm - hi);
            bk[SUB] = hi;
            bk[SUB + 1] = mid;
            bk[SUB + 2] = tf32_trunc(nrm - hi - mid);
        } else {
            bk[SUB] = __int_as_float(0x7f800000);  // padding never screens in
        }
#pragma unroll
        for (int kb = 0; kb < kKB; ++kb) {
            float4 *dst = reinterpret_cast<float4 *>(sb + ((c >> 3) * (kKB * 128) + kb * 128 + (c & 7) * 16) / 4);
            if (span_ok(dst, 16, sb, kSbBytes, 16)) *dst = make_float4(bk[4 * kb], bk[4 * kb + 1], bk[4 * kb + 2], bk[4 * kb + 3]);
        }
        if constexpr (kNB == 2) {
            // second piece: -2c's next 11 bits, nothing in the constant columns
            float *sb2 = sb + 256 * L::kRowBytes / 4;
#pragma unroll
            for (int kb = 0; kb < kKB; ++kb) {
                float4 *dst = reinterpret_cast<float4 *>(sb2 + ((c >> 3) * (kKB * 128) + kb * 128 + (c & 7) * 16) / 4);
                if (span_ok(dst, 16, sb, kSbBytes, 16))
                    *dst = kb < SUB / 4 ? make_float4(bm[4 * kb], bm[4 * kb + 1], bm[4 * kb + 2], bm[4 * kb + 3])
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (c < n_pad) {
            float *ex = sx + (c / kGC) * L::kGroupFloats + ((c % kGC) >> 1) * (2 * SUB) + (c & 1);
#pragma unroll
            for (int i = 0; i < SUB; ++i)
                if (span_ok(ex + 2 * i, 4, sx, sx_bytes, 4)) ex[2 * i] = real ? -v[i] : __int_as_float(0x7fc00000);
        }
        // maxima over the block's centroids: warp reduction, then one atomic per
        // warp (nonnegative floats, and NaN above +inf, order as their bits)
        const uint32_t mn = __reduce_max_sync(0xffffffffu, real ? __float_as_uint(nrm) : 0u);
        if (lane == 0) atomicMax(&smax[0], mn);
#pragma unroll
        for (int i = 0; i < SUB; ++i) {
            const uint32_t ma = __reduce_max_sync(0xffffffffu, real ? __float_as_uint(fabsf(v[i])) : 0u);
            if (lane == 0) atomicMax(&smax[1 + i], ma);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const float c2 = __uint_as_float(smax[0]);
    // A_i, floored at 2^-100 (compared as bits, so a NaN maximum stays NaN):
    // the floor covers the tiny-codebook terms the tensor core may flush
    float amax[SUB];
#pragma unroll
    for (int i = 0; i < SUB; ++i) amax[i] = __uint_as_float(max(smax[1 + i], 0x0d800000u));
    // 2 eps_tc + 2 gamma_SUB; with split rows, 2 (1 + 2^-9) eps_tc and the
    // dropped low part's 2^-19; with split codebooks too, 2^-17 for the three
    // dropped products
    const float kBtc = (kNA == 2 ? 2.00390625f : 2.0f) * 1.5258789e-5f + 2.0f * gamma_u(SUB) +
                       (kF32 ? 7.6293945e-6f : kNA == 2 ? 1.9073486e-6f : 0.0f);
    const float kD = 4.0f * gamma_u(SUB + 2);
    const float kTiny = 7.8886091e-31f;  // 2^-100
    // this thread's accumulator: lane rt, the NCOL columns of tile th
    const uint32_t lane_base = ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(th * NCOL);
    const uint32_t sa_addr = smem_addr(sa), sb_addr = smem_addr(sb);
    constexpr uint32_t kSbo = kKB * 128;

    // this thread's row of the first tile
    float xr[SUB];
    auto load_x = [&](int64_t row, float (&v)[SUB]) {
        if (row < n_per_group && VQ_VSPAN(xg + (size_t)row * SUB, SUB, x, nx, kRowAlign)) {
            load_row<T, SUB>(xg + (size_t)row * SUB, v);
            smooth_row<SUB, SMOOTH>(v, sg, row, smooth_ns);
        } else {
#pragma unroll
            for (int i = 0; i < SUB; ++i) v[i] = 0.f;
        }
    };
    load_x(th < tiles_per_block ? row_base + (int64_t)th * 128 + rt : n_per_group, xr);

    uint32_t phase = 0;
    bool alive = true;  // block-wide: every wait so far completed within POLLS polls
    // this thread's waits: kWaitLate, kWaitFailed; thread 0 also keeps, in
    // bits 2-3, one more than the parity of the last phase it started (0: none)
    uint32_t wst = 0;
    const int steps = (tiles_per_block + TPS - 1) / TPS;
    for (int step = 0; step < steps; ++step) {
        const int tile = step * TPS + th;  // this thread's tile; past tiles_per_block: none
        const bool own = tile < tiles_per_block;
        const int64_t row = own ? row_base + (int64_t)tile * 128 + rt : n_per_group;
        if (row_base + (int64_t)step * TPS * 128 >= n_per_group) break;  // block-uniform

        // A rows of this tile (the MMA of the previous tile has completed)
        if constexpr (kNA == 2) {
            float pc3[2][SUB];
#pragma unroll
            for (int i = 0; i < SUB; ++i) {
                pc3[0][i] = tf32_trunc(xr[i]);
                pc3[1][i] = tf32_trunc(xr[i] - pc3[0][i]);  // of the exact low bits of xr[i]
            }
#pragma unroll
            for (int pc = 0; pc < 2; ++pc)
#pragma unroll
                for (int kb = 0; kb < SUB / 4; ++kb) {
                    float4 *dst = reinterpret_cast<float4 *>(sa + (th * 2 + pc) * (L::kABytes / 4) +
                                                             ((rt >> 3) * (kKB * 128) + kb * 128 + (rt & 7) * 16) / 4);
                    if (span_ok(dst, 16, sa, kSaBytes, 16))
                        *dst = make_float4(pc3[pc][4 * kb], pc3[pc][4 * kb + 1], pc3[pc][4 * kb + 2], pc3[pc][4 * kb + 3]);
                }
        } else {
#pragma unroll
            for (int kb = 0; kb < SUB / 4; ++kb) {
                float4 *dst = reinterpret_cast<float4 *>(sa + th * (L::kABytes / 4) +
                                                         ((rt >> 3) * (kKB * 128) + kb * 128 + (rt & 7) * 16) / 4);
                if (span_ok(dst, 16, sa, kSaBytes, 16)) *dst = make_float4(xr[4 * kb], xr[4 * kb + 1], xr[4 * kb + 2], xr[4 * kb + 3]);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        float gmin[kNG];
#pragma unroll
        for (int k = 0; k < kNG; ++k) gmin[k] = __int_as_float(0x7f800000);
#pragma unroll
        for (int pass = 0; pass < 256 / NCOL; ++pass) {
            const int c0 = pass * NCOL;
            if (c0 >= n_pad) break;  // block-uniform
            const int ncols = n_pad - c0 < NCOL ? n_pad - c0 : NCOL;
            if constexpr (POLLS < kWaitPolls) {
                // a wait that gave up but completed (possible only when POLLS
                // is below the full limit): this pass's phase without an MMA
                if (tid == 0 && (wst & (kWaitLate | kWaitFailed)) == kWaitLate) {
                    (void)mbar_arrive(bar);
                    wst = (wst & 3u) | ((phase + 1u) << 2);
                }
            }
            if (tid == 0 && !(wst & kWaitLate)) {  // never a second phase outstanding
                const uint32_t idesc = umma_idesc_tf32((uint32_t)ncols);
#pragma unroll
                for (int h = 0; h < TPS; ++h) {  // the step's tiles, each into its NCOL columns
                    // (A piece, B piece) products: (hi, hi), (mid, hi), (hi, mid)
#pragma unroll
                    for (int pp = 0; pp < kNA + kNB - 1; ++pp) {
                        const uint32_t pa = (uint32_t)(h * kNA) + (pp == 1 && kNA == 2 ? 1u : 0u);
                        const uint32_t pb = pp == kNA ? 1u : 0u;
#pragma unroll
                        for (int kstep = 0; kstep < kK / 8; ++kstep) {
                            const uint64_t ad =
                                umma_smem_desc(sa_addr + pa * (uint32_t)L::kABytes + kstep * 256, 128, kSbo);
                            const uint64_t bd = umma_smem_desc(
                                sb_addr + pb * (uint32_t)(256 * L::kRowBytes) + (c0 >> 3) * kSbo + kstep * 256, 128, kSbo);
                            // the bytes the two operands span (16 or ncols / 8
                            // groups of 8 rows, kSbo apart, 256 bytes each) and
                            // the accumulator columns
                            const bool op_ok =
                                span_ok(sa + (pa * L::kABytes + kstep * 256) / 4, 15 * kSbo + 256, sa, kSaBytes, 16) &&
                                span_ok(sb + (pb * 256 * L::kRowBytes + (c0 >> 3) * kSbo + kstep * 256) / 4,
                                        (ncols / 8 - 1) * kSbo + 256, sb, kSbBytes, 16) &&
                                index_ok(h * NCOL + ncols - 1, NCOL * TPS);
                            if (op_ok) umma_tf32(tmem + (uint32_t)(h * NCOL), ad, bd, idesc, pp > 0 || kstep > 0);
                        }
                    }
                }
                umma_commit(bar);
                wst = (wst & 3u) | ((phase + 1u) << 2);
            }
            // a wait that gives up is agreed on once per tile, below; the
            // scores of that tile are never used, but are read only once the
            // MMA is done
            wst |= mbar_wait_state<POLLS>(bar, phase);
            phase ^= 1u;
            tc_fence_after();
            if (NCOL == 64 && ncols == 64) {  // block-uniform
                uint32_t v[64];
                tmem_load32_async(tmem + lane_base, v);
                tmem_load32_async(tmem + lane_base + 32u, v + 32);
                tmem_wait_ld(v);
#pragma unroll
                for (int q = 0; q < 64 / kGC; ++q) gmin[c0 / kGC + q] = group_min<kGC>(v + q * kGC);
            } else {
#pragma unroll
                for (int j = 0; j < NCOL; j += 32) {
                    if (j < ncols) {  // block-uniform
                        uint32_t v[32];
                        tmem_load32_async(tmem + lane_base + (uint32_t)j, v);
                        tmem_wait_ld(v);
#pragma unroll
                        for (int q = 0; q < 32 / kGC; ++q) gmin[(c0 + j) / kGC + q] = group_min<kGC>(v + q * kGC);
                    }
                }
            }
            tc_fence_before();
            __syncthreads();  // tensor memory is read before the next MMA writes it
            tc_fence_after();
        }

        // next tile's row, in flight during the bookkeeping below
        float xn[SUB];
        load_x(tile + TPS < tiles_per_block ? row + TPS * 128 : n_per_group, xn);

        // ---- bound, candidate groups, exact re-evaluation
        const float m1 = tree_min<kNG>(gmin);
        float sabs = 0.f, xx = 0.f;
#pragma unroll
        for (int i = 0; i < SUB; ++i) {
            sabs = fmaf(fabsf(xr[i]), amax[i], sabs);
            xx = fmaf(xr[i], xr[i], xx);
        }
        const float base = c2 + sabs;
        const float bnd = kBtc * base + kTiny;
        const float dmax = fmaxf(0.f, xx + m1 + bnd);
        const float thr = m1 + (2.0f * bnd + kD * dmax + kTiny);
        const bool ok = base < 1e30f && dmax < 1e37f;
        // candidate groups: gmin[k] <= thr exactly when fl(thr - gmin[k]) has a
        // clear sign bit (rounding keeps the sign of the exact difference and
        // gives +0 for equal operands); groups past the codebook hold +inf.
        // The sign bits are gathered with one funnel shift per group.
        uint32_t out_bits = 0;
#pragma unroll
        for (int k = kNG - 1; k >= 0; --k)
            out_bits = __funnelshift_l(__float_as_uint(__fsub_rn(thr, gmin[k])), out_bits, 1);
        const uint32_t mask = ~out_bits & (kNG == 32 ? 0xffffffffu : (1u << kNG) - 1u);
        const int cnt = __popc(mask);
        const int ga = __ffs(mask) - 1;
        const int gb = cnt > 1 ? __ffs(mask & (mask - 1)) - 1 : -1;
        if (tid == 0) *qcount = 0u;
        if (!__syncthreads_and(!(wst & kWaitLate))) {
            // a wait gave up: wait once more, with the full limit, for the
            // last phase thread 0 started (the only one that can be
            // outstanding) before the accumulator memory is freed; record the
            // tile
            alive = false;
            if (tid == 0) {
                if (wst >> 2) (void)mbar_wait<kWaitPolls>(bar, (wst >> 2) - 1u);
                *qcount = (uint32_t)step;
                raise_status(kStatusWaitGaveUp);
            }
            break;
        }
#ifdef VQ_TC_STATS
        if (row < n_per_group) {
            float excl = __int_as_float(0x7f800000);
#pragma unroll
            for (int k = 0; k < kNG; ++k)
                if (!((mask >> k) & 1u)) excl = fminf(excl, gmin[k]);
            const bool tight = excl - thr <= bnd;
            const int b = !ok || cnt > 2 || cnt == 0 ? 4 : (cnt - 1) * 2 + (tight ? 1 : 0);
            atomicAdd(&g_tc_stats[b], 1ull);
        }
#endif
        uint32_t id = 0;
        if (!ok || cnt > 2 || cnt == 0) {
            id = kQueued;
            if (row < n_per_group) {
                const uint32_t k = atomicAdd(qcount, 1u);
                if (VQ_SPAN(queue + k, 1, queue, THREADS)) queue[k] = (uint32_t)tid;
            }
        } else {
            // exact distances, two centroids per packed evaluation, ascending
            // index with a strict "<" (lowest index wins ties)
            float2 xx[SUB];
#pragma unroll
            for (int i = 0; i < SUB; ++i) xx[i] = make_float2(xr[i], xr[i]);
            const float2 one2 = make_float2(one, one);
            float best = __int_as_float(0x7f800000);
            for (int pass = 0; pass < 2; ++pass) {
                const int gsel = pass == 0 ? ga : gb;
                if (gsel < 0) break;
                const float *gp = sx + gsel * L::kGroupFloats;  // per-lane group: divergent reads
#pragma unroll 4
                for (int pr = 0; pr < kGC / 2; ++pr) {
                    float2 nc[SUB];
#pragma unroll
                    for (int k = 0; k < SUB / 2; ++k) {
                        const float4 *src = reinterpret_cast<const float4 *>(gp + pr * 2 * SUB + 4 * k);
                        const float4 q = span_ok(src, 16, sx, sx_bytes, 16) ? *src : make_float4(0.f, 0.f, 0.f, 0.f);
                        nc[2 * k] = make_float2(q.x, q.y);
                        nc[2 * k + 1] = make_float2(q.z, q.w);
                    }
                    const float2 dd = pair_dist<SUB>(xx, nc, one2);
                    const uint32_t c0 = (uint32_t)(gsel * kGC + 2 * pr);
                    if (dd.x < best) {
                        best = dd.x;
                        id = c0;
                    }
                    if (dd.y < best) {
                        best = dd.y;
                        id = c0 + 1;
                    }
                }
            }
        }
        if (row < n_per_group && id != kQueued && VQ_SPAN(og + row, 1, out, nout)) store_index(og + row, id);
        __syncthreads();

        // ---- queued rows of this tile: one warp per row, exact scan
        const uint32_t nq = *qcount;
        for (uint32_t q = (uint32_t)warp; q < nq; q += THREADS / 32) {
            if (!VQ_SPAN(queue + q, 1, queue, THREADS)) break;  // warp-uniform
            const uint32_t qt = queue[q];  // the queued row's thread: tile qt >> 7 of the step, row qt & 127
            const int64_t qrow = row_base + (int64_t)(step * TPS + (int)(qt >> 7)) * 128 + (qt & 127);
            if (!VQ_SPAN(xg + (size_t)qrow * SUB, SUB, x, nx)) continue;  // warp-uniform
            float xq[SUB];
#pragma unroll
            for (int i = 0; i < SUB; ++i) xq[i] = widen(xg[(size_t)qrow * SUB + i]);
            smooth_row<SUB, SMOOTH>(xq, sg, qrow, smooth_ns);
            float best = __int_as_float(0x7f800000);
            uint32_t bi = kQueued;
            for (int c = lane; c < n_centroids; c += 32) {
                const float *cp = sx + (c / kGC) * L::kGroupFloats + ((c % kGC) >> 1) * (2 * SUB) + (c & 1);
                float nc[SUB];
#pragma unroll
                for (int i = 0; i < SUB; ++i) nc[i] = span_ok(cp + 2 * i, 4, sx, sx_bytes, 4) ? cp[2 * i] : 0.f;
                const float d = one_dist<SUB>(xq, nc, one);
                if (d < best) {
                    best = d;
                    bi = (uint32_t)c;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ob = __shfl_xor_sync(0xffffffffu, best, off);
                const uint32_t oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ob < best || (ob == best && oi < bi)) {
                    best = ob;
                    bi = oi;
                }
            }
            if (lane == 0 && VQ_SPAN(og + qrow, 1, out, nout)) store_index(og + qrow, bi == kQueued ? 0u : bi);
        }
#pragma unroll
        for (int i = 0; i < SUB; ++i) xr[i] = xn[i];
        // the __syncthreads at the top of the next tile orders queue reuse
    }

    tc_fence_before();
    __syncthreads();
    if (!alive) {
        // a wait gave up: mark the rows of the failed step and of every later one
        for (int st = (int)*qcount; st < steps; ++st) {
            const int t = st * TPS + th;
            const int64_t r = row_base + (int64_t)t * 128 + rt;
            if (t < tiles_per_block && r < n_per_group && VQ_SPAN(og + r, 1, out, nout)) store_index(og + r, kQueued);
        }
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NCOL * TPS));
}

}  // namespace vqk
