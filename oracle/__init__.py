"""fp64 CPU oracle (test infrastructure; never imported by the product path)."""
from .attention import (MASK_ADD, attn_bwd_ref, attn_fwd_ref, attn_key_cols_ref,  # noqa: F401
                        attn_probs_ref, attn_rows_ref)
