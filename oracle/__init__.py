"""CPU oracle for the multi-LoRA MoE adapter path (test infrastructure only).

Only tests/, the package smoke check and the benchmark's CPU-baseline leg may
import this package.  It does not import the product package, and the product
package does not import it.
"""
from .oracle import (align, align_plain, fused, fused_sampled, fused_ex, capacity_tokens, capacity_blocks,  # noqa: F401
                     STATUS_BAD_EXPERT_ID, STATUS_BAD_LORA_ID, STATUS_CAPACITY)
