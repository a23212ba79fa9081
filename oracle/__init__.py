"""fp64 CPU oracles: test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import it; the
CUDA product path never does. attn_ref.py covers causal (GQA) attention; seqtile_ref.py
covers the sequence-tiled readout + cross-entropy loss and the SwiGLU MLP.
"""
from .attn_ref import (attn_bwd_ref, attn_bwd_trunked_ref, attn_dkdv_window_ref,  # noqa: F401
                       attn_fwd_ref, attn_fwd_trunked_ref, attn_group_from_stats_ref,
                       attn_group_ref, attn_row_stats_ref, attn_rows_ref)
from .seqtile_ref import (ce_loss_bwd_ref, ce_loss_ref, ce_rows_ref, mlp_bwd_ref,  # noqa: F401
                          mlp_ref, mlp_rows_ref)
