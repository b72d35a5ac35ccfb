"""GB300-native continuous-batched transformer decode (decode_step_batch).

The compute path is the CUDA library ``_build/libfs.so`` (C ABI in
``include/fs.h``); ``fs`` is its thin Python binding, ``synth`` the seeded
synthetic input generators, ``build`` the nvcc build step.
"""

__all__ = ["build", "fs", "synth"]
