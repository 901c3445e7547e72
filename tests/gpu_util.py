"""Helpers shared by the GPU parity tests (no arithmetic of the method)."""
import os

import numpy as np
import torch

# max|err| / max|ref| bounds (bf16 outputs; fp32-accumulated adapter grads)
TOL_BF16 = 2e-2
TOL_F32 = 5e-3


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def dump(name: str, **arrays):
    """With LORA_DEBUG_DUMP=<dir>, save arrays for offline inspection."""
    d = os.environ.get("LORA_DEBUG_DUMP")
    if not d:
        return
    os.makedirs(d, exist_ok=True)
    np.savez_compressed(os.path.join(d, name + ".npz"),
                        **{k: (np64(v) if isinstance(v, torch.Tensor) else np.asarray(v))
                           for k, v in arrays.items()})


def cuda(t: torch.Tensor) -> torch.Tensor:
    return t.to("cuda").contiguous()
