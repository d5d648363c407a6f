"""Multi-LoRA batched linear layer for GB300 (sm_103a).

The compute lives in ``liblora.so`` (hand-written CUDA behind a C ABI,
declared in ``include/lora.h``).  ``lora_serving_device_gb300.lora`` is the
thin ctypes binding; ``workloads`` draws seeded synthetic inputs.
Submodules are imported on first use so that drawing inputs never needs the
compiled library.
"""
import importlib

__all__ = ["lora", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
