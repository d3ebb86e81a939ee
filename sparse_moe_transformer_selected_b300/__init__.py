"""B300-native gpt-oss MoE MLP block.

The compute lives in the CUDA library libmoe_b300.so (C ABI declared in
include/moe.h).  `sparse_moe_transformer_selected_b300.moe` is the thin Python
binding with the same entry-point names; `inputs` draws seeded synthetic
workloads.  Importing the package does not load the library; the first call
through the binding does, and raises if it is missing.
"""
