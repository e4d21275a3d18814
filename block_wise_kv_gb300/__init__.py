"""GB300 (sm_103a) per-layer inner denoising step of block-wise diffusion-LLM
decoding: fused RMSNorm + QKV + RoPE + paged KV write, block attention, and
the exact FACache state merge, behind a small C ABI (include/dllm.h).

Importing the package loads nothing; ``block_wise_kv_gb300.dllm`` loads the
CUDA library and fails loudly if it has not been built.
"""
__all__ = ["inputs", "dllm"]
