"""GB300-native KV-cache compression: fused smoothing + randomized Hadamard +
group-wise min-max quantization + bit-packing, and a chunked lossless stage
pipeline, behind the C ABI of include/kvc.h (libkvc.so, CUDA for sm_103a)."""
__all__ = ["kvc", "codec", "synth", "workloads", "build"]
