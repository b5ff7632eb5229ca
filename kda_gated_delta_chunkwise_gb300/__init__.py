"""KDA (Kimi Delta Attention) gated-delta recurrence for GB300 (sm_103a).

Per sequence and head, S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1}
+ beta_t k_t v_t^T and o_t = S_t^T q_t (the web page
"研究KimiK3，我发现大模型正在学会“管理自己的计算”", pwwt.cn, §四 and §二.1).

Entry points (thin ctypes binding over the C ABI in include/kda.h):
``prefill`` (per-channel, scalar or no gate), ``prefill_fp8`` (MX-style FP8
q, k, v), ``prefill_segmented`` (one long sequence cut into segments that run
at once), ``varlen_prefill``,
``decode_step``; host (CPU) tensors given to ``prefill`` or ``prefill_fp8``
go through the native host-buffer pipeline (kda_prefill_host,
kda_prefill_fp8_host); and for serving with a pool of states indexed by slot:
``varlen_prefill_slots``, ``decode_step_slots``; for training,
``prefill_backward`` (the gradients of ``prefill``). Build the CUDA library with
``kda_gated_delta_chunkwise_gb300.build.build()`` first.
"""
from ._binding import (ALGOS, EXPORTS, GATES, KDA_DEV_BAD_CU_SEQLENS, KDA_DEV_BAD_SLOT,  # noqa: F401
                       KDA_DEV_OK, KdaError, decode_step, decode_step_slots, device_errors, lib_path, load,
                       prefill, prefill_backward, prefill_fp8, prefill_segmented, prefill_segmented_workspace_bytes,
                       prefill_workspace_bytes, segment_plan, selftest_bounded_wait, varlen_prefill,
                       varlen_prefill_backward,
                       varlen_prefill_slots, varlen_workspace_bytes)
