"""Fused vocabulary-row losses (cross-entropy, top-k distillation KL, teacher top-k) for GB300.

The compute path is the C-ABI library ``libvloss.so`` (CUDA, sm_103a), built
in-tree from ``csrc/``; ``top_kl_distill_gb300.vloss`` is its Python binding.
"""
__all__ = ["vloss", "workloads", "slicing"]
