"""Qwen3-0.6B-style decoder forward for one GB300 (sm_103a): a C-ABI CUDA library and its binding.

Submodules: ``binding`` (ctypes calls of libqwen3_gb300.so and a device-memory owner),
``build`` (nvcc build of the library), ``synth`` (seeded synthetic weights and tokens).
Importing the package loads nothing; ``binding.load_library()`` loads the CUDA library and
fails if it has not been built.
"""
