"""GB300-native per-frame decode step of a Moshi-style RQ-Transformer.

The compute lives in a C-ABI CUDA library (csrc/, include/rq.h) built for sm_103a;
`binding` is its ctypes binding, `configs` the model shapes and `synth` the seeded
synthetic inputs.  Importing the package loads nothing native.
"""
