"""GB300-native multi-LoRA Mixture-of-Experts adapter path.

Two stages, both CUDA kernels for sm_103a behind a C-ABI library
(include/moe_lora.h):
  * moe_lora_align: per active LoRA slot, count (token, top-k) pairs per
    expert, pad to block_size, prefix-sum and scatter them in order;
  * moe_lora_fused_shrink_expand: y[m,k,:] (+)= (x[m] A[l,e]^T) B[l,e]^T with
    the rank-r intermediate kept on chip.

The Python binding (lora_moe_gb300.binding) only marshals arguments; importing
this package loads nothing.
"""

__all__ = ["binding", "inputs"]
