"""GB300-native CREDIT reduce-reuse library: clustered DSMEM row softmax,
LayerNorm and RMSNorm behind a C ABI (libcredit.so), with a thin ctypes
binding.  The compute path runs only in the library's CUDA kernels."""
