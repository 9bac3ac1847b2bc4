"""Float64 CPU oracle (test infrastructure only; see attn_ref and attn_bwd_ref)."""
from .attn_ref import (  # noqa: F401
    attention_fwd, attention_fwd_jagged, attention_fwd_jvp, attention_fwd_jvp_jagged,
    attention_fwd_jvp_rows, default_scale, head_fwd, head_fwd_jvp, to_f64,
)
from .attn_bwd_ref import attention_bwd, attention_bwd_jagged, head_bwd  # noqa: F401,E402
