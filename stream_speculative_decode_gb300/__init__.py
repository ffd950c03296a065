"""Segmented speculative-verify step (LFM2 shared-round decode with drafts) for
NVIDIA GB300 (sm_103a).

  tf      ctypes binding of libtf.so (the C ABI of include/tf.h); importing it
          without a built library raises ImportError -- there is no fallback
  step    device buffers, segment table and the whole verify step on a CUDA
          stream (optionally one CUDA graph)
  inputs  seeded synthetic workloads
  build   nvcc build of libtf.so for sm_103a
"""
