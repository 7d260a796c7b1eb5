"""Forward pass of one Mixture-of-Experts layer on a GB300 (sm_103a).

The compute lives in the C-ABI library ``libmoe.so`` (CUDA kernels, see
``include/moe.h``); ``top_routing_grouped_02_gb300.moe`` is the thin Python
binding over it. ``synth`` draws the seeded synthetic inputs.
"""
