"""Exact scaled-dot-product attention for sm_103a (B300) behind a C ABI.

The computation lives in the CUDA library built from ``csrc/`` (see
``include/attn.h``); ``binding`` marshals PyTorch tensors into it and
``workloads`` draws the seeded synthetic inputs. Importing the package does
not load the library; the first call through ``binding`` does, and fails
loudly if it is missing.
"""
__all__ = ["binding", "workloads", "build"]
