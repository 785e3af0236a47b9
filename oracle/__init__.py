"""CPU oracle (test infrastructure only; never on the product path)."""

from .paged_attention import (  # noqa: F401
    OracleInputError,
    append,
    append_vllm_layout,
    blocked_from_vllm_layout,
    decode,
    decode_fast,
    decode_vllm_layout,
    gather_rows,
    kv_head_of,
    softmax,
    varlen,
    varlen_fast,
    varlen_vllm_layout,
)
