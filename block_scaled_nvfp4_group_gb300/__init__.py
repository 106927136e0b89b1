"""NVFP4 grouped GEMM for GB300 (sm_103a).

The product is the C-ABI library built from ``csrc/`` (declared in
``include/nvfp4_group_gemm.h``); ``ops`` marshals PyTorch tensors into it and
``workloads`` draws seeded synthetic inputs.  Importing the package does not
load the CUDA library; the first call into ``ops`` does, and raises if the
library is missing.
"""

__all__ = ["ops", "workloads", "device"]


def __getattr__(name):
    if name in ("ops", "workloads", "device", "_abi", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
