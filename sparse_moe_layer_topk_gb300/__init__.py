"""GB300-native (sm_103a) hot path of a LatentMoE sparse expert layer.

The compute lives in libmoe.so (CUDA, C ABI declared in include/moe.h);
`_lib` binds it with ctypes under the same names, `layer` strings the calls
into a full forward / backward, `inputs` draws the seeded synthetic inputs.
Importing the package does not load the library; the first call does, and it
raises if libmoe.so has not been built.
"""
__all__ = ["_lib", "inputs", "layer", "build"]
