"""GB300-native MoE FusedDispatch / FusedCombine on one GPU.

The compute path is the CUDA library ``libmoe`` (sm_103a kernels behind a
C ABI, declared in ``include/moe.h``); ``combine_moe_plan_gb300.moe`` is its
thin ctypes binding.  ``combine_moe_plan_gb300.workloads`` draws the seeded
synthetic inputs.  Importing the package loads nothing; the binding loads the
library on first use and raises if it has not been built.
"""
