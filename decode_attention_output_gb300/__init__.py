"""decode_attention_output_gb300: one decode step of grouped-query attention plus
the output projection, as hand-written sm_103a CUDA kernels behind a C ABI.

The compute entry points (``decode_attn_fwd``, ``decode_attn_only``, their
``_paged`` forms over a block-table cache and ``_fp8`` forms over an e4m3 cache, ``decode_attn_only_noalloc``,
``decode_attn_scores``, ``decode_attn_oproj``) live in :mod:`.binding`, which
loads ``_lib/libdecode_attn.so`` on first use and raises if it is missing.
:mod:`.synth` holds the seeded synthetic input generators and the workload
table; it imports nothing else from the package.
"""
from .binding import (  # noqa: F401
    EXPORTS,
    DecodeAttnError,
    da_tensor_t,
    decode_attn_device_error,
    decode_attn_fwd,
    decode_attn_fwd_fp8,
    decode_attn_fwd_paged,
    decode_attn_get_option,
    decode_attn_last_device_error,
    decode_attn_only,
    decode_attn_only_fp8,
    decode_attn_only_noalloc,
    decode_attn_only_paged,
    decode_attn_oproj,
    decode_attn_release,
    decode_attn_scores,
    decode_attn_set_option,
    describe,
    load,
    status_str,
)
