"""The all-to-all of compressed batch slices on three gloo ranks (CPU): every
rank splits its batch of its own tables into one container per destination
(the oracle's chunked buffer stands in for the codec here), the ranks trade
sizes and containers with error_bounded_lossy_gb300.exchange, and every
receiver restores each sender's tables into its columns of one output
("Accelerating Communication in Deep Learning Recommendation Model Training
with Dual-Level Adaptive Lossy Compression", §III-A stages 2 and 3, §III-E
Fig. 7).  The assembled output must equal, bit for bit, the senders' own
reconstructions of that slice."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

TABLES = (2, 3, 1)      # tables owned by ranks 0, 1, 2
B, D = 300, 16


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _batch(rank):
    import workloads
    wl = workloads.make("tiny", batch=B, tables=TABLES[rank], seed=rank)
    return wl.x.numpy(), wl.eb.numpy()


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from error_bounded_lossy_gb300.exchange import exchange_containers
        x, eb = _batch(rank)
        buf, offs = oracle.compress_chunked(x, eb, world)
        recv, roffs = exchange_containers(torch.from_numpy(buf), torch.from_numpy(offs.astype(np.int64)))
        ro = roffs.tolist()
        b0, b1 = oracle.chunk_rows(B, world)[rank]
        out = np.full((b1 - b0, sum(TABLES), D), np.float32(-1.0))
        col = 0
        ok = all(o % 16 == 0 for o in ro)
        for s in range(world):
            cont = recv[ro[s]:ro[s + 1]].numpy()
            oracle.decompress_columns(cont, b1 - b0, TABLES[s], D, sum(TABLES), col, out=out)
            # what sender s reconstructs of this slice of its own batch
            xs, ebs = _batch(s)
            sbuf, soffs = oracle.compress_chunked(xs, ebs, world)
            want = oracle.decompress_chunked(sbuf, soffs, B, TABLES[s], D)[b0:b1]
            ok = ok and np.array_equal(out[:, col:col + TABLES[s]].view(np.uint32), want.view(np.uint32))
            col += TABLES[s]
        q.put((rank, ok, ro))
    except Exception as e:   # reported to the parent, which fails the test
        q.put((rank, False, repr(e)))
    dist.barrier()
    dist.destroy_process_group()


def test_three_ranks_exchange_and_assemble():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = len(TABLES)
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    for rank, ok, detail in res:
        assert ok, (rank, detail)
    assert all(p.exitcode == 0 for p in procs)
