"""CPU float64 oracle for Ring Attention's blockwise exact attention.

Test infrastructure only: the tests, the smoke check and the bench's CPU
baseline leg may use it; the product path never does.
"""
from .attention import (  # noqa: F401
    below_or_on_diag,
    ref_bwd,
    ref_bwd_head_blocked,
    ref_fwd,
    ref_fwd_rows,
    ref_probs,
    ref_ring_fwd,
    visible,
)
from .decode import (  # noqa: F401
    decode_visible,
    filled_lengths,
    ref_decode,
    ref_decode_rows,
    ref_ring_decode,
)
from .ffn import ffn_rows, ref_blockwise_ffn  # noqa: F401
