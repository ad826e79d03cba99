/*
 * vq_encode.h -- C ABI of the GB300 product-vector-quantisation encoder.
 *
 * The operation ("quantize_vq"): each key vector of the KV cache is split into
 * sub-vectors of length sub_dim, and each sub-vector is encoded as the index
 * of its nearest centroid in a codebook of n_centroids rows, by squared L2
 * distance.  Source: "I Wrote a Metal Kernel to Stop My Mac From OOMing",
 * section "What Even Is a KV Cache" (steps 1-3: split into sub-vectors, a
 * K-means codebook, encode each sub-vector as its nearest centroid's index)
 * and section "The Kernel: 18 Lines of MSL" (the exact arithmetic):
 *
 *   dist(c) = sum over i = 0 .. sub_dim-1, in ascending i, of
 *             (float(x[i]) - float(codebook[c][i]))^2
 *   evaluated in IEEE fp32 with round-to-nearest: the subtraction, the square
 *   and the running sum each round separately (never fused into an FMA);
 *   out = the smallest c whose dist(c) is minimal (a strict "<" running
 *   argmin from (+inf, 0)); NaN distances never win; a row whose distances
 *   are all NaN or +inf encodes to 0; denormals are kept.
 *
 * Results are bit-exact against that definition: no approximation, no
 * tolerance.  The [N, n_centroids, sub_dim] difference tensor of the
 * straightforward implementation ("What quantize_vq Was Doing Wrong") is
 * never materialised; the library allocates no device or host memory.
 *
 * Common rules for every entry point below:
 *   - All array pointers are DEVICE pointers owned by the caller, row-major
 *     and contiguous.  x and the codebook(s) share one element type
 *     (vq_dtype).  out_idx must not overlap the inputs.
 *   - The call validates its arguments on the host and returns an error
 *     status before launching anything.  On success the work is enqueued on
 *     `stream` (0 = the legacy default stream) and the call returns without
 *     synchronising; results are valid once the stream has reached that
 *     point.
 *   - A launch failure returns VQ_ERR_CUDA; the CUDA error is left for the
 *     caller to inspect (cudaGetLastError) and is not cleared.
 *   - The tensor-core kernel waits for its matrix units with a bounded
 *     number of polls.  Should a wait give up (never observed in normal
 *     use), the rows the block has not encoded are written as 0xFFFFFFFF, an
 *     index no codebook has, and the device status word records it
 *     (vq_kernel_status, VQ_KSTATUS_WAIT_GAVE_UP); with 8-bit codes the
 *     marker is 255, a valid code when n_centroids is 256, so there only the
 *     status word tells.
 *   - N = 0 (or n_per_group = 0) is valid: VQ_OK, nothing is launched, and
 *     the pointers may be NULL.
 *   - Supported shapes: 1 <= sub_dim <= 32, 1 <= n_centroids <= 4096.
 *     sub_dim 4 and 8 with x aligned to sub_dim * element size take the
 *     fast kernels; other shapes and misaligned x take a general kernel that
 *     produces the same indices.
 *   - Thread safety: calls may be made from several host threads; the
 *     library keeps only a per-device cache of attributes, filled on first
 *     use.
 */
#ifndef VQ_ENCODE_H
#define VQ_ENCODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; declared opaquely so this header needs no CUDA headers. */
typedef struct CUstream_st *vq_stream_t;

typedef enum {
    VQ_OK = 0,
    VQ_ERR_INVALID_ARG = 1, /* null pointer with work to do, negative size, unknown dtype */
    VQ_ERR_UNSUPPORTED = 2, /* sub_dim or n_centroids outside the supported range */
    VQ_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    VQ_ERR_INTERNAL = 4     /* a broken internal invariant (should not happen) */
} vq_status;

/* Element type shared by x and the codebook(s). */
typedef enum {
    VQ_F16 = 0,  /* IEEE binary16 */
    VQ_BF16 = 1, /* bfloat16 */
    VQ_F32 = 2   /* IEEE binary32 */
} vq_dtype;

/*
 * vq_encode -- encode N sub-vectors against one codebook.
 *   x          [n][sub_dim]            device, dtype
 *   codebook   [n_centroids][sub_dim]  device, dtype
 *   out_idx    [n]                     device, uint32, written
 * The call is asynchronous on `stream`.
 */
vq_status vq_encode(const void *x, const void *codebook, int64_t n, int32_t n_centroids,
                    int32_t sub_dim, vq_dtype dtype, uint32_t *out_idx, vq_stream_t stream);

/*
 * vq_encode_grouped -- encode n_groups independent slices, each with its own
 * codebook, in one launch (e.g. one codebook per layer, or per (layer, KV
 * head), for a cache laid out [layers][batch, heads, tokens, head_dim]).
 *   x          [n_groups][n_per_group][sub_dim]       device, dtype
 *   codebooks  [n_groups][n_centroids][sub_dim]       device, dtype
 *   out_idx    [n_groups][n_per_group]                device, uint32, written
 * Row r of group g is encoded against codebooks[g] only.  n_groups = 1 is the
 * same as vq_encode.  The call is asynchronous on `stream`.
 */
vq_status vq_encode_grouped(const void *x, const void *codebooks, int64_t n_groups,
                            int64_t n_per_group, int32_t n_centroids, int32_t sub_dim,
                            vq_dtype dtype, uint32_t *out_idx, vq_stream_t stream);

/*
 * vq_encode_grouped_host -- the same encode for inputs and outputs in HOST
 * memory; returns once out_host holds the indices (it synchronises `stream`).
 *   x_host, codebooks_host, out_host    host memory, same layouts as above
 *   x_dev        >= n_groups*n_per_group*sub_dim elements, device, scratch
 *   codebooks_dev >= n_groups*n_centroids*sub_dim elements, device, scratch
 *   out_dev      >= n_groups*n_per_group uint32, device, scratch
 * If x_host and out_host are page-locked (pinned) memory the GPU can address,
 * the kernel reads x and writes the indices directly across the CPU-GPU link
 * (on GB300 the coherent NVLink-C2C) while it computes: only the codebooks
 * are copied (to codebooks_dev), and x_dev / out_dev are not touched.
 * Otherwise x is copied to x_dev and the indices back from out_dev, in chunks
 * on two internal copy streams that overlap the encode of neighbouring chunks
 * when the input is large.  The internal streams and events are created on
 * the first such call on a device and kept until exit; host calls on one
 * device are serialised by a lock.  The device buffers are the caller's; the
 * library allocates no memory.
 */
vq_status vq_encode_grouped_host(const void *x_host, const void *codebooks_host,
                                 int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                                 int32_t sub_dim, vq_dtype dtype, uint32_t *out_host,
                                 void *x_dev, void *codebooks_dev, uint32_t *out_dev,
                                 vq_stream_t stream);

/*
 * vq_encode_grouped_u8 -- vq_encode_grouped writing 8-bit codes: the same
 * indices, one byte each ("What Even Is a KV Cache": 16 indices at 8 bits
 * each for a 128-dim key, the 16x compression).  Requires n_centroids <= 256
 * (VQ_ERR_UNSUPPORTED otherwise).
 *   out_idx    [n_groups][n_per_group]   device, uint8, written
 * Same arguments, rules and asynchrony as vq_encode_grouped.
 */
vq_status vq_encode_grouped_u8(const void *x, const void *codebooks, int64_t n_groups,
                               int64_t n_per_group, int32_t n_centroids, int32_t sub_dim,
                               vq_dtype dtype, uint8_t *out_idx, vq_stream_t stream);

/*
 * vq_encode_grouped_smooth -- the grouped encode fused with per-channel
 * smoothing of the keys ("VecInfer -- 16x with Metal acceleration": per-channel
 * smooth scaling tames the outlier channels that defeat plain VQ).  Each
 * element is divided by its channel's factor in fp32, rounded to nearest, and
 * the divided row is encoded by the exact formula of vq_encode (same indices
 * as encoding the divided rows).  The query side is the caller's: attention
 * over these codes takes the query multiplied by the same factors.
 *   x          [n_groups][n_per_group][sub_dim]   device, dtype; row m of a
 *              group holds channels (m % (head_dim / sub_dim)) * sub_dim + i
 *              of a key vector, so n_per_group is a multiple of
 *              head_dim / sub_dim
 *   smooth     [n_groups][head_dim]               device, fp32 factors
 *   codebooks  [n_groups][n_centroids][sub_dim]   device, dtype
 *   out_idx    [n_groups][n_per_group]            device, uint32 (index_bytes
 *              4) or uint8 codes (index_bytes 1, n_centroids <= 256)
 * sub_dim 4 or 8 and x aligned to its row (up to 16 bytes), else
 * VQ_ERR_UNSUPPORTED.  Other rules and asynchrony as vq_encode_grouped.
 */
vq_status vq_encode_grouped_smooth(const void *x, const float *smooth, const void *codebooks,
                                   int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                                   int32_t sub_dim, int32_t head_dim, vq_dtype dtype, void *out_idx,
                                   int32_t index_bytes, vq_stream_t stream);

/*
 * vq_dequantize_grouped -- decode ("dequantize_vq"): rebuild each sub-vector
 * as a copy of its codebook row ("I Wrote a Metal Kernel to Stop My Mac From
 * OOMing", section "Mistake 1: I Wrote the Dequant Kernel First": indices in,
 * reconstructed vectors out, a gather).
 *   idx        [n_groups][n_per_group]              device, uint32 (index_bytes
 *                                                   = 4) or uint8 (index_bytes = 1)
 *   codebooks  [n_groups][n_centroids][sub_dim]     device, dtype
 *   out        [n_groups][n_per_group][sub_dim]     device, dtype, written
 * out[g][m][:] = codebooks[g][idx[g][m]][:] bit for bit; an index outside
 * [0, n_centroids) writes a row of zeros.  Same pointer, size and error rules
 * as vq_encode_grouped (index_bytes other than 1 or 4: VQ_ERR_INVALID_ARG);
 * asynchronous on `stream`.
 */
vq_status vq_dequantize_grouped(const void *idx, int32_t index_bytes, const void *codebooks,
                                int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                                int32_t sub_dim, vq_dtype dtype, void *out, vq_stream_t stream);

/*
 * vq_attention_decode -- attention of one decode query per (batch, query
 * head) over a KV cache held as 8-bit product-VQ codes, without rebuilding the
 * keys or values ("I Wrote a Metal Kernel to Stop My Mac From OOMing",
 * section "What's Next: Phase 2": the per-query LUT q @ codebook^T, scores by
 * LUT lookup, softmax-weighted value sum in one fused pass).
 *   q            [batch][heads_q][head_dim]                 device, dtype
 *   k_codes      [batch][heads_kv][tokens][head_dim/sub_dim] device, uint8
 *   k_codebooks  [heads_kv][n_centroids][sub_dim]           device, dtype
 *   v_codes, v_codebooks                                    same, for values
 *   out          [batch][heads_q][head_dim]                 device, dtype, written
 *   workspace    >= vq_attention_workspace_bytes(...) bytes, device, 16-byte
 *                aligned, scratch owned by the caller (smaller: fewer token
 *                slices are used, down to one; too small for one: error)
 * Query head h uses KV head h / (heads_q / heads_kv) (grouped-query
 * attention).  With K^[t] and V^[t] the codebook rows the codes select:
 *   out = softmax_t(scale * q . K^[t]) @ V^[t]
 * over the last `window` tokens (0: all tokens); scale <= 0 means
 * 1/sqrt(head_dim).  Accumulation is fp32; no tokens gives zeros.
 * Requirements: heads_q % heads_kv == 0, head_dim % sub_dim == 0,
 * sub_dim % 4 == 0, head_dim <= 512, head_dim/sub_dim in {4, 8, 16, 32, 64},
 * n_centroids <= 256, code arrays aligned to min(head_dim/sub_dim, 16) bytes
 * (VQ_ERR_INVALID_ARG / VQ_ERR_UNSUPPORTED otherwise).  Asynchronous on
 * `stream`; the library allocates nothing.
 */
vq_status vq_attention_decode(const void *q, const uint8_t *k_codes, const void *k_codebooks,
                              const uint8_t *v_codes, const void *v_codebooks, int64_t batch,
                              int32_t heads_q, int32_t heads_kv, int64_t tokens, int32_t head_dim,
                              int32_t sub_dim, int32_t n_centroids, int64_t window, float scale,
                              vq_dtype dtype, void *out, void *workspace, size_t workspace_bytes,
                              vq_stream_t stream);

/* Workspace vq_attention_decode uses for these sizes on the current device
 * (0 for invalid sizes). */
size_t vq_attention_workspace_bytes(int64_t batch, int32_t heads_q, int32_t heads_kv,
                                    int64_t tokens, int32_t head_dim, int32_t sub_dim,
                                    int32_t n_centroids, int64_t window);

/* Bytes of device scratch built into the library for
 * vq_attention_decode_static. */
#define VQ_ATTN_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * vq_attention_decode_static -- vq_attention_decode without a workspace
 * argument: the partials go to an array of VQ_ATTN_STATIC_SCRATCH_BYTES
 * (8 MiB) that the library holds in device memory for each device.  The pages
 * have no counterpart; this is an interface for callers that cannot allocate
 * device memory per call: a decode loop whose HBM is fully planned up front
 * (the quantised KV cache takes what the weights leave), or plain C host code
 * with no caching allocator, for which a cudaMalloc / cudaFree per decode step
 * would synchronise the device.  The call allocates nothing.
 * Arguments, layouts and results are those of vq_attention_decode.  When the
 * partials of the shape's default plan need more than the array holds, fewer
 * token slices are used; a shape whose single slice,
 * batch * heads_q * (head_dim + 2) * 4 bytes, exceeds the array returns
 * VQ_ERR_INVALID_ARG.  Every call on a device shares the one array: calls whose
 * kernels overlap on the GPU (on different streams, or from several host
 * threads without ordering between them) race on it and give wrong results,
 * so issue them in one stream order.  Nothing in the array needs clearing.
 * Device: the array used is the CURRENT device's; `stream` and every pointer
 * must belong to that device (a q on another device returns
 * VQ_ERR_INVALID_ARG).  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) and keeps it: make that first call
 * before any stream capture, and do not call cudaDeviceReset on a device
 * between calls (the kept address would then be stale).
 */
vq_status vq_attention_decode_static(const void *q, const uint8_t *k_codes,
                                     const void *k_codebooks, const uint8_t *v_codes,
                                     const void *v_codebooks, int64_t batch, int32_t heads_q,
                                     int32_t heads_kv, int64_t tokens, int32_t head_dim,
                                     int32_t sub_dim, int32_t n_centroids, int64_t window,
                                     float scale, vq_dtype dtype, void *out, vq_stream_t stream);

/*
 * Sibling encoders on the same nearest-centroid rule (the page of five
 * hand-tuned Metal compute kernels for TurboQuant, "Kernel 2: Scalar Quantize
 * / Dequantize" and "Kernel 3: Fused Hadamard + Quantize").  One fp32
 * codebook `centroids` [n_centroids] (1..256, device) serves every element;
 * indices are uint8.
 *
 * vq_scalar_quantize -- out[e] = the j minimising fl(fl(float(x[e]) -
 * centroids[j])^2), lowest j on ties, NaN never winning, 0 when nothing wins.
 *   x          [n]  device, dtype
 *   out        [n]  device, uint8, written
 *   workspace  device scratch of the caller, 16-byte aligned.  fp16 input
 *              with 2, 4, 8 or 16 centroids does not use it: each block
 *              builds a 2 KiB table of the 1,024 buckets of fp16 patterns
 *              (top 10 bits) from the codebook's cut points, and looks every
 *              key up there.  Other fp16 / bf16 input with at least
 *              vq_scalar_quantize_workspace_bytes (65536) bytes evaluates the
 *              rule once for each of the 65,536 input bit patterns, and the
 *              pass becomes a table lookup.  Otherwise (fp32 input, or NULL /
 *              smaller workspace) every element scans the codebook.  The
 *              indices are the same on every path.
 */
size_t vq_scalar_quantize_workspace_bytes(vq_dtype dtype);
vq_status vq_scalar_quantize(const void *x, vq_dtype dtype, int64_t n, const float *centroids,
                             int32_t n_centroids, uint8_t *out, void *workspace,
                             size_t workspace_bytes, vq_stream_t stream);

/*
 * vq_scalar_dequantize -- out[e] = centroids[idx[e]] rounded to nearest in the
 * output dtype (the page's half(centroids[idx])); an index >= n_centroids
 * gives 0.  idx [n] uint8, out [n] dtype, both device.
 */
vq_status vq_scalar_dequantize(const uint8_t *idx, int64_t n, const float *centroids,
                               int32_t n_centroids, vq_dtype dtype, void *out,
                               vq_stream_t stream);

/*
 * vq_hadamard_rotate -- randomised Hadamard rotation of each row of dim
 * elements (dim a power of two, 1..1024): v = float(x) * diag (fp32); for
 * stride = 1, 2, ..., dim/2 every pair (e, e + stride) with e % (2 stride) <
 * stride becomes (v[e] + v[e+stride], v[e] - v[e+stride]); y = v * s with s
 * the fp32 value of 1/sqrt(dim) (correctly rounded).  Every step is one
 * rounded fp32 operation in exactly this order.
 *   x     [n_rows][dim]  device, dtype, aligned to min(dim/32 elements, 16
 *         bytes) (one element for dim <= 32)   diag  [dim]  device, fp32
 *   y     [n_rows][dim]  device, fp32, written
 * vq_hadamard_quantize -- the same rotation fused with vq_scalar_quantize of
 * every rotated value; out [n_rows][dim] uint8 (4-byte aligned when dim >=
 * 128).  Neither writes the rotated keys to memory in the fused form.
 */
vq_status vq_hadamard_rotate(const void *x, vq_dtype dtype, const float *diag, int64_t n_rows,
                             int32_t dim, float *y, vq_stream_t stream);
vq_status vq_hadamard_quantize(const void *x, vq_dtype dtype, const float *diag, int64_t n_rows,
                               int32_t dim, const float *centroids, int32_t n_centroids,
                               uint8_t *out, vq_stream_t stream);

/*
 * Multi-GPU partition of one encode job.  Every row of a grouped encode is
 * independent ("What Even Is a KV Cache": each sub-vector is encoded on its
 * own against its codebook), so a job [n_groups][n_per_group] splits across
 * `world` GPUs with no exchange: each rank encodes the rows it owns against
 * replicated codebooks and keeps their indices.
 *
 * vq_partition -- the rows rank `rank` of `world` owns: one contiguous range
 * of the flattened row index g * n_per_group + m, [floor(rank T / world),
 * floor((rank + 1) T / world)) with T = n_groups * n_per_group (the ranks'
 * shares differ by at most one row; every row is owned exactly once), cut
 * into at most three slices, in row order, that each is one grouped encode:
 * rows [row, row + n_rows) of each of the groups [group, group + n_groups).
 * A slice with n_groups > 1 covers whole groups (row 0, n_rows =
 * n_per_group); the others lie in one group.  Its encode is
 * vq_encode_grouped(x + (group * n_per_group + row) * sub_dim,
 * codebooks + group * n_centroids * sub_dim, n_groups, n_rows, ...), whose
 * indices are the next n_groups * n_rows of the rank's share.
 *   slices     [3] host memory, written (the first *n_slices)
 *   n_slices   host, written: 0 to 3 (0: the rank owns no row)
 * world < 1, rank outside [0, world), negative sizes or NULL pointers:
 * VQ_ERR_INVALID_ARG.  Host arithmetic only: no device is needed.
 */
typedef struct {
    int64_t group;    /* first group */
    int64_t n_groups; /* groups */
    int64_t row;      /* first row within each of them */
    int64_t n_rows;   /* rows of each group */
} vq_slice;

vq_status vq_partition(int64_t n_groups, int64_t n_per_group, int32_t world, int32_t rank,
                       vq_slice *slices, int32_t *n_slices);

/* Static, human-readable text for a status code (never NULL). */
const char *vq_status_string(vq_status status);

/*
 * vq_describe_launch -- which kernel and launch shape vq_encode_grouped would
 * use for these arguments on the current device, as NUL-terminated text in
 * buf (truncated to buflen).  Performs no launch.  Returns the same
 * argument errors as vq_encode_grouped.
 */
vq_status vq_describe_launch(int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                             int32_t sub_dim, vq_dtype dtype, const void *x, char *buf,
                             int32_t buflen);

/*
 * vq_kernel_status -- the out-of-band failure record of the library's
 * kernels on the current device.  Waits for the device to finish all work
 * (cudaDeviceSynchronize), then sets *bits to the OR of the status bits that
 * kernels launched on this device have set since the last clear, and resets
 * them to zero if `clear` is nonzero.  0 means every kernel finished its work
 * normally.  A bit is needed beside the in-band marker because the marker of
 * 8-bit codes (255) is a valid code when n_centroids is 256.
 *   VQ_KSTATUS_WAIT_GAVE_UP   a tensor-core encode's wait for its matrix
 *                             units gave up; the rows it had not encoded hold
 *                             0xFFFFFFFF (255 as 8-bit codes)
 *   VQ_KSTATUS_OUT_OF_BOUNDS  bounds-checked build only: an index fell
 *                             outside its buffer and the access was skipped
 * Returns VQ_ERR_INVALID_ARG for a NULL `bits`, VQ_ERR_CUDA if the
 * synchronisation or the read fails (*bits is then 0).  Not part of the
 * pages' method; it is this library's failure report.
 */
#define VQ_KSTATUS_WAIT_GAVE_UP 0x1u
#define VQ_KSTATUS_OUT_OF_BOUNDS 0x2u
vq_status vq_kernel_status(uint32_t *bits, int32_t clear);

/* ABI version of this header (bumped on incompatible changes). */
#define VQ_ENCODE_ABI_VERSION 1
int32_t vq_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VQ_ENCODE_H */
