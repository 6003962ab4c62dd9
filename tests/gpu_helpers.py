"""GPU-side helpers for the parity tests: every kernel runs through the C ABI
(via the package's ctypes binding); inputs come from the seeded generator."""
import numpy as np
import torch

from paged_kv_cache_97_gb300.batch import DecodeBatch, bits_of, dev_pool, to_dev_bf16  # noqa: F401

GpuStep = DecodeBatch


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
