// vq_attn.cu -- C ABI entry points of decode attention over product-VQ codes
// (see include/vq_encode.h for the contract of each function).
//
// Host side only: validate arguments, plan the launch (query heads per
// block, token runs per block), launch the partial and combine kernels of
// vq_attn.cuh on the caller's stream.  The library allocates no memory: the
// partials go to the caller's workspace.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "vq_encode.h"
#include "vq_attn.cuh"
#include "vq_host.h"
#include "vq_status.cuh"

VQH_STATUS_READER(vqh_status_attn)

namespace {

size_t elem_size(vq_dtype d) { return d == VQ_F32 ? 4 : 2; }

int device_sms() { return vqh_device_sms(); }

struct AttnPlan {
    vqk::AttnShape sh;
    int gpb;  // query heads per block
    size_t smem;
    size_t part_bytes_per_split;
    int64_t base;  // blocks per split: batch * heads_kv * head groups
};

constexpr int kAttnThreads = vqk::kAttnThreads;
constexpr size_t kAttnMaxSmem = 200 * 1024;
constexpr size_t kSmemPerSm = 228 * 1024;  // shared memory per SM, 1 KiB of it per block reserved

bool attn_ns_supported(int ns) { return ns == 4 || ns == 8 || ns == 16 || ns == 32 || ns == 64; }

vq_status attn_validate(int64_t batch, int32_t heads_q, int32_t heads_kv, int64_t tokens,
                        int32_t head_dim, int32_t sub_dim, int32_t n_centroids, int64_t window)
{
    if (batch < 0 || tokens < 0 || window < 0) return VQ_ERR_INVALID_ARG;
    if (heads_q < 1 || heads_kv < 1 || heads_q % heads_kv) return VQ_ERR_INVALID_ARG;
    if (sub_dim < 1 || head_dim < 1 || head_dim % sub_dim) return VQ_ERR_INVALID_ARG;
    if (head_dim > 512 || sub_dim % vqk::kAttnVw || !attn_ns_supported(head_dim / sub_dim))
        return VQ_ERR_UNSUPPORTED;
    if (n_centroids < 1 || n_centroids > 256) return VQ_ERR_UNSUPPORTED;
    return VQ_OK;
}

// Query heads per block: the largest of 8, 4, 2, 1 that divides the GQA ratio
// and whose shared memory fits.  Chunk runs (splits): the count that
// minimises waves * (chunks per run + the ~0.7 chunk a block spends on its
// tables and the final merge).
vq_status attn_plan(int64_t batch, int32_t heads_q, int32_t heads_kv, int64_t tokens,
                    int32_t head_dim, int32_t sub_dim, int32_t n_centroids, int64_t window,
                    float scale, int elem, AttnPlan *p)
{
    const int qpk = heads_q / heads_kv;
    const int ns = head_dim / sub_dim;
    int gpb = 0;
    for (int g = 8; g >= 1; g /= 2)
        if (qpk % g == 0 && vqk::attn_smem(g, ns, sub_dim, elem).total <= kAttnMaxSmem) {
            gpb = g;
            break;
        }
    if (gpb == 0) return VQ_ERR_UNSUPPORTED;
    const vqk::AttnSmem lay = vqk::attn_smem(gpb, ns, sub_dim, elem);
    const size_t smem = lay.total;
    // the queries are staged in the value-codebook region before it is filled
    if (((size_t)gpb * head_dim + (size_t)4 * ns) * sizeof(float) > lay.pw - lay.vcb)
        return VQ_ERR_INTERNAL;
    const int chunk = vqk::attn_chunk(ns);
    const int64_t first = window > 0 && window < tokens ? tokens - window : 0;
    const int64_t chunks = (tokens - first + chunk - 1) / chunk;
    const int64_t base = batch * heads_kv * (qpk / gpb);
    const int sms = device_sms() > 0 ? device_sms() : 152;
    int64_t per_sm = (int64_t)(kSmemPerSm / (smem + 1024));
    if (per_sm > 2048 / kAttnThreads) per_sm = 2048 / kAttnThreads;
    if (per_sm < 1) per_sm = 1;
    const int64_t slots = sms * per_sm;
    int64_t best = 1;
    double best_cost = 1e300;
    const int64_t max_splits = chunks < 4096 ? chunks : 4096;
    for (int64_t k = 1; k <= max_splits && base > 0; ++k) {
        const int64_t waves = (base * k + slots - 1) / slots;
        const double cost = (double)waves * ((double)((chunks + k - 1) / k) + 0.7);
        if (cost < best_cost) {
            best_cost = cost;
            best = k;
        }
    }
    p->sh = vqk::AttnShape{batch, heads_q, heads_kv, head_dim, sub_dim, n_centroids, tokens, first,
                           chunks, (int32_t)best,
                           (scale > 0.f ? scale : 1.0f / sqrtf((float)head_dim)) *
                               1.4426950408889634f};
    p->gpb = gpb;
    p->smem = smem;
    p->part_bytes_per_split = (size_t)batch * heads_q * (head_dim + 2) * sizeof(float);
    p->base = base;
    return VQ_OK;
}

template <typename T, int NS, int GPB, int VW>
vq_status attn_launch_k(const AttnPlan &p, const void *q, const uint8_t *kcodes, const void *kcb,
                        const uint8_t *vcodes, const void *vcb, float *part, cudaStream_t st)
{
    auto kp = vqk::attn_partial<T, NS, GPB, VW>;
    if (p.smem > 48 * 1024 &&
        cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) !=
            cudaSuccess)
        return VQ_ERR_CUDA;
    kp<<<(unsigned)(p.base * p.sh.splits), kAttnThreads, p.smem, st>>>(
        static_cast<const T *>(q), kcodes, static_cast<const T *>(kcb), vcodes,
        static_cast<const T *>(vcb), p.sh, part);
    return vqh_launched(st, vqh_status_attn);
}

template <typename T, int NS, int VW>
vq_status attn_launch_vw(const AttnPlan &p, const void *q, const uint8_t *kcodes, const void *kcb,
                         const uint8_t *vcodes, const void *vcb, float *part, cudaStream_t st)
{
    switch (p.gpb) {
    case 1: return attn_launch_k<T, NS, 1, VW>(p, q, kcodes, kcb, vcodes, vcb, part, st);
    case 2: return attn_launch_k<T, NS, 2, VW>(p, q, kcodes, kcb, vcodes, vcb, part, st);
    case 4: return attn_launch_k<T, NS, 4, VW>(p, q, kcodes, kcb, vcodes, vcb, part, st);
    case 8: return attn_launch_k<T, NS, 8, VW>(p, q, kcodes, kcb, vcodes, vcb, part, st);
    }
    return VQ_ERR_INTERNAL;
}

template <typename T, int NS>
vq_status attn_launch_ns(const AttnPlan &p, const void *q, const uint8_t *kcodes, const void *kcb,
                         const uint8_t *vcodes, const void *vcb, float *part, cudaStream_t st)
{
    if constexpr (sizeof(T) == 2) {
        if (vqk::attn_vw(p.sh.sub_dim, 2) == 8)
            return attn_launch_vw<T, NS, 8>(p, q, kcodes, kcb, vcodes, vcb, part, st);
    }
    return attn_launch_vw<T, NS, vqk::kAttnVw>(p, q, kcodes, kcb, vcodes, vcb, part, st);
}

template <typename T>
vq_status attn_launch(const AttnPlan &p, const void *q, const uint8_t *kcodes, const void *kcb,
                      const uint8_t *vcodes, const void *vcb, void *out, float *part,
                      cudaStream_t st)
{
    vq_status s = VQ_ERR_INTERNAL;
    switch (p.sh.head_dim / p.sh.sub_dim) {
    case 4: s = attn_launch_ns<T, 4>(p, q, kcodes, kcb, vcodes, vcb, part, st); break;
    case 8: s = attn_launch_ns<T, 8>(p, q, kcodes, kcb, vcodes, vcb, part, st); break;
    case 16: s = attn_launch_ns<T, 16>(p, q, kcodes, kcb, vcodes, vcb, part, st); break;
    case 32: s = attn_launch_ns<T, 32>(p, q, kcodes, kcb, vcodes, vcb, part, st); break;
    case 64: s = attn_launch_ns<T, 64>(p, q, kcodes, kcb, vcodes, vcb, part, st); break;
    }
    if (s != VQ_OK) return s;
    const int64_t rows = p.sh.batch * p.sh.heads_q;
    const int threads = (p.sh.head_dim + 31) / 32 * 32;
    // a programmatic dependent of the partials' launch: its blocks are
    // scheduled as the partial blocks retire and wait on the device for
    // the whole partial grid (griddepcontrol.wait), instead of a full launch
    // gap after it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, vqk::attn_combine<T>, (const float *)part, rows, p.sh.head_dim,
                           p.sh.splits, static_cast<T *>(out)) != cudaSuccess) {
        (void)cudaGetLastError();
        return VQ_ERR_CUDA;
    }
    return vqh_launched(st, vqh_status_attn);
}

// Scratch of vq_attention_decode_static: the per-slice partials live in this
// one array instead of a caller workspace.  Nothing in it has to start at
// zero (every partial the merge reads is written earlier in the same call).
// All calls on a device share it.
static __device__ __align__(256) unsigned char g_attn_scratch[VQ_ATTN_STATIC_SCRATCH_BYTES];

// Device address of g_attn_scratch on the current device, looked up on the
// first call on that device and kept (a cudaDeviceReset between calls would
// leave it stale, which the header rules out); nullptr if the lookup fails.
// `dev` is the current device.
void *static_scratch(int dev)
{
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" {

size_t vq_attention_workspace_bytes(int64_t batch, int32_t heads_q, int32_t heads_kv,
                                    int64_t tokens, int32_t head_dim, int32_t sub_dim,
                                    int32_t n_centroids, int64_t window)
{
    if (attn_validate(batch, heads_q, heads_kv, tokens, head_dim, sub_dim, n_centroids, window) !=
        VQ_OK)
        return 0;
    size_t most = 0;
    for (int elem = 2; elem <= 4; elem += 2) {  // the plan of 16-bit and of fp32 inputs
        AttnPlan p;
        if (attn_plan(batch, heads_q, heads_kv, tokens, head_dim, sub_dim, n_centroids, window,
                      0.f, elem, &p) != VQ_OK)
            return 0;
        const size_t bytes = p.part_bytes_per_split * (size_t)p.sh.splits;
        if (bytes > most) most = bytes;
    }
    return most;
}

vq_status vq_attention_decode(const void *q, const uint8_t *k_codes, const void *k_codebooks,
                              const uint8_t *v_codes, const void *v_codebooks, int64_t batch,
                              int32_t heads_q, int32_t heads_kv, int64_t tokens, int32_t head_dim,
                              int32_t sub_dim, int32_t n_centroids, int64_t window, float scale,
                              vq_dtype dtype, void *out, void *workspace, size_t workspace_bytes,
                              vq_stream_t stream)
{
    if (dtype != VQ_F16 && dtype != VQ_BF16 && dtype != VQ_F32) return VQ_ERR_INVALID_ARG;
    vq_status s = attn_validate(batch, heads_q, heads_kv, tokens, head_dim, sub_dim, n_centroids,
                                window);
    if (s != VQ_OK) return s;
    if (batch == 0) return VQ_OK;
    const size_t es = elem_size(dtype);
    if (!q || !k_codebooks || !v_codebooks || !out || !workspace) return VQ_ERR_INVALID_ARG;
    if (tokens > 0 && (!k_codes || !v_codes)) return VQ_ERR_INVALID_ARG;
    const uintptr_t code_align = head_dim / sub_dim < 16 ? head_dim / sub_dim : 16;
    if ((uintptr_t)q % es || (uintptr_t)k_codebooks % es || (uintptr_t)v_codebooks % es ||
        (uintptr_t)out % es || (uintptr_t)workspace % 16 || (uintptr_t)k_codes % code_align ||
        (uintptr_t)v_codes % code_align)
        return VQ_ERR_INVALID_ARG;
    AttnPlan p;
    if ((s = attn_plan(batch, heads_q, heads_kv, tokens, head_dim, sub_dim, n_centroids, window,
                       scale, (int)es, &p)) != VQ_OK)
        return s;
    // fewer token slices if the workspace holds fewer partials
    const int64_t fit = (int64_t)(workspace_bytes / p.part_bytes_per_split);
    if (fit < 1) return VQ_ERR_INVALID_ARG;
    if (fit < p.sh.splits) p.sh.splits = (int32_t)fit;
    if (p.base * p.sh.splits > 0x7fffffffLL || p.sh.batch * p.sh.heads_q > 0x7fffffffLL)
        return VQ_ERR_UNSUPPORTED;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *part = static_cast<float *>(workspace);
    switch (dtype) {
    case VQ_F16: return attn_launch<__half>(p, q, k_codes, k_codebooks, v_codes, v_codebooks, out, part, st);
    case VQ_BF16:
        return attn_launch<__nv_bfloat16>(p, q, k_codes, k_codebooks, v_codes, v_codebooks, out,
                                          part, st);
    case VQ_F32: return attn_launch<float>(p, q, k_codes, k_codebooks, v_codes, v_codebooks, out, part, st);
    }
    return VQ_ERR_INTERNAL;
}

vq_status vq_attention_decode_static(const void *q, const uint8_t *k_codes,
                                     const void *k_codebooks, const uint8_t *v_codes,
                                     const void *v_codebooks, int64_t batch, int32_t heads_q,
                                     int32_t heads_kv, int64_t tokens, int32_t head_dim,
                                     int32_t sub_dim, int32_t n_centroids, int64_t window,
                                     float scale, vq_dtype dtype, void *out, vq_stream_t stream)
{
    vq_status s = attn_validate(batch, heads_q, heads_kv, tokens, head_dim, sub_dim, n_centroids,
                                window);
    if (s != VQ_OK) return s;
    if (batch == 0) return VQ_OK;
    // one token slice of partials must fit in the array
    if ((uint64_t)batch * (uint64_t)heads_q * (uint64_t)(head_dim + 2) * sizeof(float) >
        VQ_ATTN_STATIC_SCRATCH_BYTES)
        return VQ_ERR_INVALID_ARG;
    // The array used is the current device's, so q must live there: a kernel
    // on another device would write the partials into this device's copy.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return VQ_ERR_CUDA;
    if (q != nullptr) {
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
            (void)cudaGetLastError();  // not a pointer CUDA knows
            return VQ_ERR_INVALID_ARG;
        }
        if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
            return VQ_ERR_INVALID_ARG;
        if (at.type == cudaMemoryTypeDevice && at.device != dev) return VQ_ERR_INVALID_ARG;
    }
    void *scratch = static_scratch(dev);
    if (scratch == nullptr) return VQ_ERR_CUDA;
    return vq_attention_decode(q, k_codes, k_codebooks, v_codes, v_codebooks, batch, heads_q,
                               heads_kv, tokens, head_dim, sub_dim, n_centroids, window, scale,
                               dtype, out, scratch, VQ_ATTN_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"
