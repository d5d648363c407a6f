"""CPU fp64 oracle (test infrastructure only; see lora_ref)."""
from .lora_ref import (  # noqa: F401
    adapter_bytes,
    build_segments,
    expand,
    lora_linear,
    lora_linear_gathered,
    lora_linear_per_request,
    lora_linear_segmented,
    lora_param_count,
    merge,
    pad_rank,
    requests_from_ids,
    shrink,
    valid_ids,
)
