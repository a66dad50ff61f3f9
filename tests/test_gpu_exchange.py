"""The exchange helper with NCCL on CUDA tensors, end to end through the codec:
a one-rank group (every call on this machine gets one GPU) compresses its batch
as a chunked buffer, trades it through error_bounded_lossy_gb300.exchange, and
restores the received container into the columns of a wider output.  The
buffer sent is compared with the oracle's chunked buffer byte for byte, the
buffer received with what was sent, and the restored columns with the oracle's
column decode bit for bit."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import error_bounded_lossy_gb300 as ebc
import oracle
import workloads
from error_bounded_lossy_gb300.exchange import exchange_containers

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_nccl_exchange_one_rank():
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    codec = ebc.Codec(0)
    try:
        wl = workloads.make("fwd", batch=1000, tables=3)
        x = wl.x.cuda()
        buf, offs = codec.compress_chunked(x, 1, wl.eb.numpy())
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        # the sending buffer is the oracle's, byte for byte, before it is exchanged
        rbuf, rofs = oracle.compress_chunked(wl.x.numpy(), wl.eb.numpy(), 1)
        assert offs.cpu().tolist() == rofs.tolist()
        assert np.array_equal(buf[: int(rofs[-1])].cpu().numpy(), rbuf)
        recv, roffs = exchange_containers(buf, offs)
        assert recv.is_cuda and roffs.tolist() == offs.tolist()
        assert np.array_equal(recv.cpu().numpy(), rbuf)
        out = torch.full((1000, 5, 128), 3.0, dtype=torch.float32, device="cuda")
        codec.decompress_columns(recv, int(roffs[-1]), 3, out, 1)
        torch.cuda.synchronize()
        assert codec.last_error() == 0
        ref = np.full((1000, 5, 128), np.float32(3.0))
        oracle.decompress_columns(recv.cpu().numpy(), 1000, 3, 128, 5, 1, out=ref)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    finally:
        codec.close()
        dist.destroy_process_group()
