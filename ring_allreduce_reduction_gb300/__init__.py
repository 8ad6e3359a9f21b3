"""vrccl: ring AllReduce over n virtual ranks resident in one GB300's HBM.

Layout:
  csrc/         C-ABI library (libvrccl.so): host side and sm_103a kernels.
  build.py      in-tree nvcc build of libvrccl.so.
  vrccl.py      Python binding with the C entry points' names (import it
                explicitly; it loads the library and fails if it is absent).
  workloads.py  seeded synthetic inputs (no reduction arithmetic).
  tune.py       measures the auto-tuning table on the GPU.

The package import itself loads nothing, so the input generator can be used
without a GPU or a built library.
"""
__all__ = ["build", "workloads"]
