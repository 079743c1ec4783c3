"""GB300-native MoE layer between DP attention and expert parallelism.

The compute path is libmoe_dp.so (hand-written sm_103a CUDA behind the C ABI
in include/moe_dp.h); ``combine_dp_gather_gb300.moe_dp`` is its Python
binding, ``combine_dp_gather_gb300.synth`` the seeded workload recipes and
``combine_dp_gather_gb300.build`` the in-tree nvcc build.  Importing the
package loads nothing; the library is loaded on first use.
"""
