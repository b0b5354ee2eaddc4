"""Device-memory plumbing: move host workloads (numpy) to CUDA tensors and back.

PyTorch serves only as the allocator and copier here; no arithmetic of the
method runs in this module.
"""
from __future__ import annotations

import dataclasses

import numpy as np


def _to_cuda_bf16(a: np.ndarray, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def _to_cuda_i32(a: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def bf16_to_host_bits(t) -> np.ndarray:
    """A CUDA bf16 tensor as host uint16 bits."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@dataclasses.dataclass
class DeviceWorkload:
    q: object
    k_cache: object
    v_cache: object
    block_tables: object
    context_lens: object
    k_new: object
    v_new: object
    slot_mapping: object


def to_device(wl, device="cuda") -> DeviceWorkload:
    return DeviceWorkload(
        q=_to_cuda_bf16(wl.q, device),
        k_cache=_to_cuda_bf16(wl.k_cache, device),
        v_cache=_to_cuda_bf16(wl.v_cache, device),
        block_tables=_to_cuda_i32(wl.block_tables, device),
        context_lens=_to_cuda_i32(wl.context_lens, device),
        k_new=_to_cuda_bf16(wl.k_new, device),
        v_new=_to_cuda_bf16(wl.v_new, device),
        slot_mapping=_to_cuda_i32(wl.slot_mapping, device),
    )


@dataclasses.dataclass
class DeviceFp8Cache:
    kv_cache: object  # uint8 e4m3 codes [num_blocks, n_kv, 2, block_size, head_dim]
    k_scale: object   # float32 [n_kv]
    v_scale: object


def fp8_to_device(c, device="cuda") -> DeviceFp8Cache:
    import torch
    return DeviceFp8Cache(
        kv_cache=torch.from_numpy(np.ascontiguousarray(c.kv_cache)).to(device),
        k_scale=torch.from_numpy(np.ascontiguousarray(c.k_scale, dtype=np.float32)).to(device),
        v_scale=torch.from_numpy(np.ascontiguousarray(c.v_scale, dtype=np.float32)).to(device))
