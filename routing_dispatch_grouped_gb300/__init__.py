"""GB300 (sm_103a) MoE expert layer: route -> dispatch -> grouped SwiGLU experts -> combine.

The compute lives in libmoe.so (CUDA kernels behind a C ABI, see include/moe.h); ``moe`` is its
thin Python binding. ``synth`` makes the seeded synthetic inputs.
"""
