"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch


def to_dev(x_u16: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit array -> CUDA bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(x_u16).view(np.int16)).view(torch.bfloat16).cuda()


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .double().numpy()


def rel_l2(got, ref) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
