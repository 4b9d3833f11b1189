"""The host side of the expert-parallel exchange on two gloo ranks (CPU only): the count
exchange and the row all-to-all give every destination the rows its sources packed for
it, sources in rank order, and the reverse exchange returns each row to its place."""
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rows(rank, n, H):
    # row i of rank r's send buffer: value 1000*r + i in every column
    return (1000 * rank + torch.arange(n, dtype=torch.float32))[:, None].repeat(1, H)


def _main(rank, world, port, counts, H, q):
    import torch.distributed as dist

    from moe_expert_ffn_03_gb300.expert_parallel import all_to_all_rows, exchange_counts
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = torch.tensor(counts[rank], dtype=torch.int32)
    send_splits, recv_splits = exchange_counts(mine)
    assert send_splits == counts[rank]
    assert recv_splits == [counts[s][rank] for s in range(world)]
    send = _rows(rank, sum(send_splits), H)
    recv = torch.empty(sum(recv_splits), H)
    all_to_all_rows(recv, send, recv_splits, send_splits)
    expect = []
    for s in range(world):
        first = sum(counts[s][:rank])
        expect.append(_rows(s, sum(counts[s]), H)[first:first + counts[s][rank]])
    ok_fwd = torch.equal(recv, torch.cat(expect))
    back = torch.empty_like(send)
    all_to_all_rows(back, recv, send_splits, recv_splits)        # the reverse exchange
    ok_back = torch.equal(back, send)
    eids = torch.arange(sum(send_splits), dtype=torch.int32)     # int32 payloads travel too
    reids = torch.empty(sum(recv_splits), dtype=torch.int32)
    all_to_all_rows(reids, eids, recv_splits, send_splits)
    q.put((rank, ok_fwd, ok_back, reids.tolist()))
    dist.destroy_process_group()


def test_two_rank_exchange_over_gloo():
    world, H = 2, 8
    counts = [[3, 5], [0, 4]]                     # rank 1 sends nothing to rank 0
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.start_processes(_main, args=(world, _free_port(), counts, H, q), nprocs=world, start_method="spawn")
    res = sorted(q.get() for _ in range(world))
    for rank, ok_fwd, ok_back, reids in res:
        assert ok_fwd and ok_back, rank
    assert res[0][3] == [0, 1, 2]                 # rank 0 received rank 0's rows 0..2, none from rank 1
    assert res[1][3] == [3, 4, 5, 6, 7, 0, 1, 2, 3]
