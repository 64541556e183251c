"""Helpers for the GPU tests: numpy <-> torch buffers with the oracle's dtypes."""

import numpy as np
import torch

TORCH = {"bf16": torch.int16, "f32": torch.float32, "bytes": torch.uint8}
NP_VIEW = {"bf16": np.int16, "f32": np.float32, "bytes": np.uint8}
NP_ORACLE = {"bf16": np.uint16, "f32": np.float32, "bytes": np.uint8}


def to_dev(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(NP_VIEW[dtype]).copy()).to(device)


def from_dev(t: torch.Tensor, dtype: str) -> np.ndarray:
    return t.cpu().numpy().view(NP_ORACLE[dtype])


def empty_dev(n: int, dtype: str, fill_byte: int = 0xA5, device="cuda") -> torch.Tensor:
    """Output buffer prefilled with a canary byte pattern (unnamed elements must keep it)."""
    t = torch.empty(n * {"bf16": 2, "f32": 4, "bytes": 1}[dtype], dtype=torch.uint8, device=device)
    t.fill_(fill_byte)
    return t.view(TORCH[dtype])


def bits_equal(a: np.ndarray, b: np.ndarray) -> bool:
    return a.shape == b.shape and np.array_equal(np.asarray(a).view(np.uint8),
                                                 np.asarray(b).view(np.uint8))
