"""Helpers for the GPU parity tests: moving oracle storage arrays (float32, or
uint16 bit patterns for fp16/bf16) to and from torch device tensors, guard
bands, and deliberately misaligned views."""
import numpy as np
import torch

F32, F16, BF16 = 0, 1, 2
TORCH_DT = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
NP_STORAGE = {F32: np.float32, F16: np.uint16, BF16: np.uint16}
CANARY = 0x5A


def to_dev(arr: np.ndarray, dt: int) -> torch.Tensor:
    arr = np.ascontiguousarray(arr)
    if dt == F32:
        return torch.from_numpy(arr.astype(np.float32, copy=False)).cuda()
    return torch.from_numpy(arr.view(np.int16)).cuda().view(TORCH_DT[dt])


def to_host(t: torch.Tensor, dt: int) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if dt == F32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


class Guarded:
    """An output tensor followed by 256 canary bytes; offset_elems shifts its
    start (to take the unaligned path)."""

    def __init__(self, numel: int, dt: int, offset_elems: int = 0):
        esz = torch.tensor([], dtype=TORCH_DT[dt]).element_size()
        self.nbytes = numel * esz
        self.off = offset_elems * esz
        self.raw = torch.full((self.off + self.nbytes + 256,), CANARY, dtype=torch.uint8,
                              device="cuda")
        self.t = self.raw[self.off:self.off + self.nbytes].view(TORCH_DT[dt])

    def canary_ok(self) -> bool:
        return bool((self.raw[self.off + self.nbytes:] == CANARY).all().item()) and \
            bool((self.raw[:self.off] == CANARY).all().item())


def misaligned_copy(t: torch.Tensor, offset_elems: int = 1) -> torch.Tensor:
    """Same values at an address offset by offset_elems elements."""
    buf = torch.empty(t.numel() + offset_elems, dtype=t.dtype, device=t.device)
    v = buf[offset_elems:]
    v.copy_(t.reshape(-1))
    return v
