"""GB300-native (sm_103a) FarSkip-Collective MoE layer stack.

The compute path is the C-ABI library ``libfs.so`` (hand-written CUDA kernels);
``fs.py`` is its thin Python binding.  ``configs.py`` and ``synth.py`` hold the
workload shapes and the seeded input generator.  Importing the package loads
nothing; ``fs.lib()`` loads the library and fails loudly when it is missing.
"""
