"""GB300 (sm_103a) ragged GQA attention with its full vector-Jacobian product.

The computation lives in ``libattn_varlen.so`` (hand-written CUDA: a device
tile scheduler, a tcgen05/TMA forward, the D = rowsum(dO * O) preprocess, and
an atomic-free backward with separate dk/dv and dq passes).  This package is
its thin binding; ``workloads`` draws seeded synthetic inputs.
"""
from .binding import (AttnError, attention_varlen_feature_full_vjp, attention_varlen_fvjp,
                      device_status, launch_count, load, workspace_size)

__all__ = ["AttnError", "attention_varlen_feature_full_vjp", "attention_varlen_fvjp",
           "device_status", "launch_count", "load", "workspace_size"]
