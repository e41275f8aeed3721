"""Independent fp64 CPU oracle (test infrastructure only; see hc_gr_oracle)."""
from .hc_gr_oracle import (  # noqa: F401
    bf16_round, sigmoid, combine, grouped_rrms, norm_weight, normalise, project, silu_h,
    up_gate, gated_mean, split_merged, merge_weight, forward, mix,
)
