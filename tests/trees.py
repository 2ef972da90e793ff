"""Seeded draft-tree inputs shared by the oracle pins and the GPU tests (the
generator lives with the other seeded inputs, in the workloads module, and
computes nothing of the op)."""
from paged_kv_attention_02_gb300.workloads import chain, mask_words, path_of, random_parents  # noqa: F401
