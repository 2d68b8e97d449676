"""fp64 CPU oracle (test infrastructure; see ``oracle.attention``)."""

from . import fp8  # noqa: F401
from .attention import (  # noqa: F401
    attention_backward,
    attention_backward_block,
    attention_backward_varlen,
    attention_forward,
    attention_forward_varlen,
    head_dkdv,
    head_dq,
    head_forward,
    head_row_stats,
    kv_head,
    tile_grid,
    valid_matrix,
)
