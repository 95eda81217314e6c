"""Paged-expert MoE layer for one GB300 (sm_103a).

A router picks top_k of E experts per token; routed experts that are not resident
are copied from a pinned host store into a per-layer K-slot GPU table (least
recently used out); the fused MoE (gate/up, SiLU*mul, down, weighted combine) then
runs over the slot table. All compute runs in the hand-written CUDA kernels of
libpagedmoe.so, reached through its C ABI (include/pagedmoe.h).
"""

from ._lib import (  # noqa: F401
    ExpertCache, PmoeError, load, moe_decode_forward_noalloc, moe_group_by_expert, moe_router_gemm_topk, moe_router_topk,
    pmoe_expert_bytes,
    PMOE_BF16, PMOE_FP8_BLOCK128, PMOE_INT4_GPTQ_G128, PMOE_MXFP4, PMOE_NVFP4, PMOE_PAGEIN_COPY_ENGINE,
    PMOE_PAGEIN_SM_PULL,
    PMOE_OK, PMOE_EINVAL, PMOE_ENOMEM, PMOE_EHOSTALLOC, PMOE_ECUDA, PMOE_EUNSUPPORTED, PMOE_ETIMEOUT,
    PMOE_EDEVICE,
)
