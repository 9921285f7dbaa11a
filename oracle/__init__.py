"""CPU fp64 oracle for the Dual-Flow decode step (test infrastructure; see dualflow_oracle)."""
from .dualflow_oracle import *  # noqa: F401,F403
from .dualflow_oracle import (DenseCache, HParams, PagedCache, attention, attention_only_step, decode_step,  # noqa: F401
                              mixture_head, rms_scale, rmsnorm, rope, round_bf16, round_f32, route, silu, softmax,
                              topk_lower_index, widen)
