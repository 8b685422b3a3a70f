"""SageAttention-style quantized attention forward for GB300 (sm_103a).

INT8 Q/K per 32-token block, FP8 E4M3 V per channel, exact integer QK^T on
the tensor cores, FP32 online softmax, FP8 P and FP32-accumulated PV, BF16
output ``[B, S, H, 128]``.  The work runs in ``libsage.so`` (C ABI in
``include/sage.h``); this package is its thin Python binding.
"""
from .sage import (EXPORTED, FAULT_ATTN_LAUNCH, FAULT_NONE, FAULT_POOL_ALLOC, FAULT_QUANT_LAUNCH,  # noqa: F401
                   HEAD_DIM, LIB_PATH, PLAN_FUSED_Q, PLAN_SMOOTH_K, Plan, SageError, attn_fwd, attn_fwd_cross, attn_fwd_launches, attn_fwd_lse,
                   attn_fwd_quantized, debug_fused_q, debug_inject_fault, debug_pool_state, debug_qk_int32,
                   debug_staging_codes, debug_wait_timeout, load_library, padded_len, quantize_qkv,
                   quantize_qkv_smooth_k, set_attention_events, set_wait_timeout_ns, sync_status,
                   workspace_bytes)
