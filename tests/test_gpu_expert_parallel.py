"""Expert parallelism on one GPU: G ranks emulated in one process (the all-to-all done by
slicing the packed buffers), and two real processes exchanging rows over gloo.

Each expert receives its rows ordered by source rank and then by token; with ranks that
hold consecutive token ranges this is the single-GPU permutation's order, so out, dx,
dprob and every expert's dW must equal the single-GPU layer's on the concatenated
tokens bit for bit.  The single-GPU layer is itself compared with the oracle in the layer
tests; out is compared with the oracle here as well.
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch

from helpers import assert_close
from moe_expert_ffn_03_gb300 import build, configs, synth
from moe_expert_ffn_03_gb300.expert_parallel import ExpertParallelFFN
from moe_expert_ffn_03_gb300.layer import ExpertFFN
from oracle import expert_ffn as ef
from oracle import routing as rt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def single_gpu(wl, inp):
    L = ExpertFFN(wl.T, wl.H, wl.I, wl.E, wl.k, training=True)
    L.quantize_weights(inp["w_gu"], inp["w_d"])
    L.forward(inp["logits"], inp["x"])
    L.backward(inp["dout"])
    torch.cuda.synchronize()
    assert L.device_error() == (0, 0)
    return L


def emulate(wl, inp, G):
    """G ranks in one process; rank r holds tokens r*T/G .. and experts r*E/G .."""
    T, El = wl.T // G, wl.E // G
    ranks = [ExpertParallelFFN(T, wl.H, wl.I, wl.E, wl.k, G, r) for r in range(G)]
    sl = lambda a, r: a[r * T:(r + 1) * T]  # noqa: E731
    for r, R in enumerate(ranks):
        R.quantize_weights(inp["w_gu"][r * El:(r + 1) * El], inp["w_d"][r * El:(r + 1) * El])
    packs = [R.dispatch_pack(sl(inp["logits"], r), sl(inp["x"], r)) for r, R in enumerate(ranks)]
    counts = np.array([p[3].cpu().tolist() for p in packs])                # [source][destination]
    send_off = np.concatenate([np.zeros((G, 1), np.int64), np.cumsum(counts, axis=1)], axis=1)
    recv_off = np.concatenate([np.zeros((1, G), np.int64), np.cumsum(counts, axis=0)], axis=0)

    def exchange(src_bufs, dst_bufs, forward):
        # forward: source s's rows for d -> d's receive buffer (sources in order);
        # back: d's rows from s -> s's return buffer (destinations in order)
        for s in range(G):
            for d in range(G):
                n = int(counts[s, d])
                a, b = int(send_off[s, d]), int(recv_off[s, d])
                if forward:
                    dst_bufs[d][b:b + n] = src_bufs[s][a:a + n]
                else:
                    dst_bufs[s][a:a + n] = src_bufs[d][b:b + n]

    for i in range(3):                                                      # x, prob, local expert id
        exchange([p[i] for p in packs], [(R.recv_x, R.recv_prob, R.recv_eid)[i] for R in ranks], True)
    backs = [R.expert_forward(int(counts[:, d].sum())) for d, R in enumerate(ranks)]
    exchange(backs, [R.ret for R in ranks], False)
    outs = [R.combine() for R in ranks]
    sends = [R.grad_pack(sl(inp["dout"], r)) for r, R in enumerate(ranks)]
    exchange(sends, [R.recv_x for R in ranks], True)
    grads = [R.expert_backward() for R in ranks]
    exchange([g[0] for g in grads], [R.ret for R in ranks], False)
    exchange([g[1] for g in grads], [R.ret_dprob for R in ranks], False)
    dxs = [R.grad_combine() for R in ranks]
    torch.cuda.synchronize()
    for R in ranks:
        assert R.device_error() == (0, 0)
    return ranks, outs, dxs


@pytest.mark.parametrize("G,dims", [(2, (384, 256, 384, 8, 2, "biased")), (4, (512, 128, 256, 8, 2, "normal")),
                                    (4, (256, 256, 128, 16, 4, "biased")), (8, (256, 128, 128, 8, 1, "normal"))])
def test_expert_parallel_emulated_equals_single_gpu(G, dims):
    wl = configs.small(*dims[:5], routing=dims[5], backward=True)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    L = single_gpu(wl, inp)
    ranks, outs, dxs = emulate(wl, inp, G)
    T, El = wl.T // G, wl.E // G
    for r, R in enumerate(ranks):
        assert torch.equal(R.idx, L.idx[r * T:(r + 1) * T])
        assert torch.equal(outs[r], L.out[r * T:(r + 1) * T])
        assert torch.equal(dxs[r][0], L.dx[r * T:(r + 1) * T])
        assert torch.equal(dxs[r][1], L.dprob[r * T:(r + 1) * T])
        assert torch.equal(R.dwgu, L.dwgu[r * El:(r + 1) * El])
        assert torch.equal(R.dwd, L.dwd[r * El:(r + 1) * El])
    # and the combined output against the oracle
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    idx, prob = rt.route_topk(inp["logits"].cpu().numpy(), wl.k)
    fwd = ef.forward(f64(inp["x"]), idx, prob.astype(np.float64), f64(inp["w_gu"]), f64(inp["w_d"]), ef.MXFP8)
    assert_close(np.concatenate([f64(o) for o in outs]), fwd["out"], "out")


def test_expert_parallel_rank_without_rows():
    """Routing that sends no token to rank 1's experts: its experts' side receives nothing,
    its weight gradients are zero, and the other rank's results still match."""
    G = 2
    wl = configs.small(256, 128, 128, 4, 1, backward=True)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    inp["logits"][:, 2:] = -50.0                                         # experts 2, 3 (rank 1) get nothing
    L = single_gpu(wl, inp)
    ranks, outs, dxs = emulate(wl, inp, G)
    assert ranks[1].n_recv == 0
    assert torch.count_nonzero(ranks[1].dwgu) == 0 and torch.count_nonzero(ranks[1].dwd) == 0
    assert torch.equal(torch.cat(outs), L.out)
    assert torch.equal(torch.cat([d[0] for d in dxs]), L.dx)


# ---- two processes on the one GPU, rows exchanged over gloo ----------------------------
def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, dims, outdir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    wl = configs.small(*dims[:5], routing=dims[5], backward=True)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    T, El = wl.T // world, wl.E // world
    R = ExpertParallelFFN(T, wl.H, wl.I, wl.E, wl.k, world, rank)
    R.quantize_weights(inp["w_gu"][rank * El:(rank + 1) * El], inp["w_d"][rank * El:(rank + 1) * El])
    out = R.forward(inp["logits"][rank * T:(rank + 1) * T], inp["x"][rank * T:(rank + 1) * T])
    dx, dprob = R.backward(inp["dout"][rank * T:(rank + 1) * T])
    torch.cuda.synchronize()
    assert R.device_error() == (0, 0)
    torch.save({k: v.cpu() for k, v in dict(out=out, dx=dx, dprob=dprob, dwgu=R.dwgu, dwd=R.dwd).items()},
               os.path.join(outdir, f"rank{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


def test_expert_parallel_two_processes_over_gloo():
    import torch.multiprocessing as mp
    dims = (384, 256, 256, 8, 2, "biased")
    world = 2
    wl = configs.small(*dims[:5], routing=dims[5], backward=True)
    inp = {k: v.cuda() for k, v in synth.make_inputs(wl, 0).items()}
    L = single_gpu(wl, inp)
    T, El = wl.T // world, wl.E // world
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(world, _free_port(), dims, d), nprocs=world, start_method="spawn")
        for r in range(world):
            got = torch.load(os.path.join(d, f"rank{r}.pt"))
            assert torch.equal(got["out"], L.out[r * T:(r + 1) * T].cpu())
            assert torch.equal(got["dx"], L.dx[r * T:(r + 1) * T].cpu())
            assert torch.equal(got["dprob"], L.dprob[r * T:(r + 1) * T].cpu())
            assert torch.equal(got["dwgu"], L.dwgu[r * El:(r + 1) * El].cpu())
            assert torch.equal(got["dwd"], L.dwd[r * El:(r + 1) * El].cpu())
