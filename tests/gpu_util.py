"""Helpers shared by the GPU parity tests (host <-> device marshalling only)."""
import numpy as np
import torch

import oracle


def dev():
    return torch.device("cuda:0")


def to_dev(a, bf16=False):
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns when bf16."""
    a = np.ascontiguousarray(a)
    if bf16:
        return torch.from_numpy(a.view(np.int16)).to(dev()).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev())


def logits_to_dev(x, dt):
    return to_dev(x, bf16=(dt == oracle.DT_BF16))


def storage_of(t):
    """CUDA tensor -> numpy in the oracle's storage convention."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


DT_OF = {"f32": oracle.DT_F32, "bf16": oracle.DT_BF16, "f16": oracle.DT_F16}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
