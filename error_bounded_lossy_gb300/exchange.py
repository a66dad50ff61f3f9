"""The all-to-all of compressed batch slices (§III-A stages 2 and 3, §III-E
"Buffer Optimization"): every rank holds one container per destination rank,
back to back in one buffer (Codec.compress_chunked); the ranks first trade the
containers' sizes, then the containers themselves, and each receiver restores
every sender's tables into its columns of one output (Codec.decompress_columns).

This module is the host side of that exchange over torch.distributed: NCCL with
CUDA tensors, gloo with CPU tensors.  It moves bytes only; the coding is the
codec's.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def exchange_containers(buf: torch.Tensor, offsets: torch.Tensor, group=None):
    """Sends container r of `buf` (bytes [offsets[r], offsets[r+1])) to rank r
    and receives one container from every rank.

    buf: uint8 tensor with the world-size containers back to back; offsets:
    int64 tensor [world + 1] on the same device.  Returns (recv, recv_offsets):
    container s of recv, bytes [recv_offsets[s], recv_offsets[s+1]), came from
    rank s.  Every container size is a multiple of 16 bytes, so each received
    container starts on a 16-byte boundary, as the decoder requires.  The split
    sizes are read on the host (an all-to-all with uneven splits needs them
    there), which synchronises the caller's stream once."""
    world = dist.get_world_size(group)
    offs = offsets.to(torch.int64)
    if offs.numel() != world + 1:
        raise ValueError(f"expected {world + 1} offsets, got {offs.numel()}")
    send_counts = offs[1:] - offs[:-1]
    recv_counts = torch.empty_like(send_counts)
    dist.all_to_all_single(recv_counts, send_counts, group=group)
    sc, rc = send_counts.tolist(), recv_counts.tolist()
    if any(c % 16 for c in sc + rc):
        raise ValueError("container sizes must be multiples of 16 bytes")
    recv = torch.empty(sum(rc), dtype=torch.uint8, device=buf.device)
    dist.all_to_all_single(recv, buf[: int(offs[-1])], rc, sc, group=group)
    recv_offsets = torch.zeros(world + 1, dtype=torch.int64, device=buf.device)
    recv_offsets[1:] = torch.cumsum(recv_counts, 0)
    return recv, recv_offsets
