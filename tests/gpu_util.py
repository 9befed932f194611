"""Helpers for the GPU parity tests: move seeded numpy inputs to the device and
read results back.  No arithmetic of the method lives here."""
import numpy as np
import torch

from diffusion_draft_tree_gb300 import workloads as wl


def dev_logits(a: np.ndarray, dtype: int, device) -> torch.Tensor:
    if dtype == wl.BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(
            torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)


def dev_bf16(a: np.ndarray, device) -> torch.Tensor:
    return dev_logits(a, wl.BF16, device)


def dev_i32(a, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)


def dev_f32(a, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def tree_to_dev(tree: dict, device) -> dict:
    out = {}
    for k, v in tree.items():
        if k == "anc_mask":
            out[k] = torch.from_numpy(np.ascontiguousarray(v).view(np.int32)).to(device)
        elif k == "score":
            out[k] = dev_f32(v, device)
        else:
            out[k] = dev_i32(v, device)
    return out
