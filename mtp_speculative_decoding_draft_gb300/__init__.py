"""MTP speculative decoding (draft chain + verification) for one GB300 GPU.

The compute runs in ``libmtpspec.so`` (CUDA, sm_103a; C ABI in
``include/mtpspec.h``); ``binding`` marshals torch CUDA tensors into its calls,
``model`` holds a device-resident draft module and its workspace, ``workloads``
draws the seeded synthetic inputs and ``metrics`` computes the acceptance
statistics.  Importing this package does not load the library; the first call
into ``binding`` does, and fails loudly if it is missing.
"""

__all__ = ["binding", "workloads", "metrics", "model", "build"]
