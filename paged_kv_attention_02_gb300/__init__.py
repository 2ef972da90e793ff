"""Paged-KV attention (`attn_paged`) for GB300 (sm_103a).

The compute path is the C-ABI library built from ``csrc/`` (declared in
``include/rad_attn.h``); ``binding`` marshals torch tensors into it.
"""
