"""GB300 (sm_103a) library for one batched speculative-speculative-decoding
round with the Saguaro algorithm: Saguaro draft sampling, lossless
verification, outcome prediction, speculation-cache lookup and tree-masked
branch attention, behind the C ABI of include/ssd.h.

``binding`` is the thin Python layer over that ABI (imported on first use so
that CPU-only tooling can import ``workloads`` without CUDA); ``workloads``
holds the seeded synthetic inputs.
"""
import importlib

__all__ = ["binding", "workloads", "build"]


def __getattr__(name):
    if name in ("binding", "workloads", "build"):
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
