"""fp64 CPU oracle for causal (GQA) attention: test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import it; the
CUDA product path never does. See attn_ref.py for what each function computes.
"""
from .attn_ref import (attn_bwd_ref, attn_bwd_trunked_ref, attn_dkdv_window_ref,  # noqa: F401
                       attn_fwd_ref, attn_fwd_trunked_ref, attn_rows_ref)
