"""Float64 CPU oracle (test infrastructure only; see attn_ref, attn_bwd_ref and attn_fp8_ref)."""
from .attn_ref import (  # noqa: F401
    attention_fwd, attention_fwd_jagged, attention_fwd_jvp, attention_fwd_jvp_jagged,
    attention_fwd_jvp_rows, default_scale, head_fwd, head_fwd_jvp, to_f64,
)
from .attn_bwd_ref import attention_bwd, attention_bwd_jagged, head_bwd  # noqa: F401,E402
from .attn_fp8_ref import attention_fwd_e5m2, e5m2_bound_terms, head_fwd_e5m2, round_e5m2  # noqa: F401,E402
