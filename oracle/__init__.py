"""CPU oracle (test infrastructure only; never on the product path)."""

from .paged_attention import (  # noqa: F401
    OracleInputError,
    append,
    decode,
    decode_fast,
    gather_rows,
    kv_head_of,
    softmax,
    varlen,
)
