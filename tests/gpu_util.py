"""Small numpy <-> torch helpers shared by the GPU tests (marshalling only)."""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def padded(rows: int, cols: int, ld: int, dtype, fill=0) -> torch.Tensor:
    """A [rows, cols] view with row stride ``ld`` into a [rows, ld] buffer."""
    buf = torch.full((rows, ld), fill, dtype=dtype, device="cuda")
    return buf[:, :cols]
