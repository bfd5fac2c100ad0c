"""GB300-native tile-based 3D Gaussian Splatting training step.

The compute path is a CUDA library for sm_103a behind a C ABI (``include/gs.h``):
``gs_project``, ``gs_bin_sort``, ``gs_raster_fused_fwd_bwd``, ``gs_grad_compact``
and ``gs_adam_deferred``.  ``differentiable_rasterizer_gb300.abi`` is the thin
ctypes binding of those calls; ``differentiable_rasterizer_gb300.pipeline`` drives
one training step with torch tensors as device memory.  ``scenes`` draws the
seeded synthetic inputs.

Importing this package does not load the CUDA library; the binding loads it on
first use and raises if it has not been built.
"""

__all__ = ["abi", "pipeline", "scenes"]
