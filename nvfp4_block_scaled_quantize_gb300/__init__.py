"""NVFP4 block-scaled quantization for one GB300 (sm_103a).

The compute path is hand-written CUDA behind the C ABI declared in ``include/nvfp4.h``;
``api`` is the thin Python binding over it (argument marshalling only). Importing the package
does not load the library: the first call into ``api`` does, and raises if it was not built.
"""
