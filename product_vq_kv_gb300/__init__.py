"""GB300-native product-vector-quantisation encoder for KV caches.

Encodes each sub-vector of a key cache as the uint32 index of its nearest
centroid (squared L2, exact fp32 arithmetic, ties to the lowest index) with
hand-written sm_103a CUDA kernels behind a C ABI (``include/vq_encode.h``).
This package is the thin Python binding of that library.
"""
from ._binding import (  # noqa: F401
    ATTN_STATIC_SCRATCH_BYTES,
    VQError,
    VQ_BF16,
    VQ_ERR_CUDA,
    VQ_ERR_INTERNAL,
    VQ_ERR_INVALID_ARG,
    VQ_ERR_UNSUPPORTED,
    VQ_F16,
    VQ_F32,
    VQ_KSTATUS_OUT_OF_BOUNDS,
    VQ_KSTATUS_WAIT_GAVE_UP,
    VQ_OK,
    load_library,
    vq_abi_version,
    vq_attention_decode,
    vq_attention_decode_static,
    vq_attention_workspace_bytes,
    vq_dequantize_grouped,
    vq_describe_launch,
    vq_encode,
    vq_encode_grouped,
    vq_encode_grouped_host,
    vq_encode_grouped_smooth,
    vq_encode_grouped_u8,
    vq_encode_partition,
    vq_hadamard_quantize,
    vq_hadamard_rotate,
    vq_kernel_status,
    vq_partition,
    vq_scalar_dequantize,
    vq_scalar_quantize,
    vq_status_string,
)
from .build import LIB_PATH  # noqa: F401
