"""spec_verify_gb300: a batched next-token sampler and speculative-decoding
verifier for NVIDIA GB300 (sm_103a).

The compute lives in libsmp.so (C ABI: include/smp.h), built in-tree by
`python -m spec_verify_gb300.build`.  `spec_verify_gb300.binding` wraps it for
PyTorch tensors; `spec_verify_gb300.workloads` makes seeded synthetic inputs.
"""

__all__ = ["binding", "build", "workloads"]
