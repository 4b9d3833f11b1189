"""Expert parallelism: the experts spread over ranks, tokens exchanged by all-to-all.

Page "英伟达开源MoE加速神器：一行代码，微调快3.7倍", section "三板斧" (expert
parallelism): the experts live on different GPUs and an All-to-All sends every
token to the GPU of its expert and brings the result back.  Page "Efficient MoE
Training for Biological Foundation Models", section "运行要求、基准与验证步骤":
the recipe runs with EP = 8 and DP x EP = #GPUs.

Layout: `world` ranks, rank r owns experts r*E/world .. (r+1)*E/world - 1 (its
local experts 0 .. E/world - 1) and holds its own T tokens.  One step of rank r:

  tokens' side   moe_route (top-k over all E experts, expert-major permutation)
                 moe_ep_pack: rows grouped by destination rank, counts per rank
  exchange       all-to-all of the counts, then of the rows (x, prob, local id)
  experts' side  moe_permute of the received rows (k = 1, their local expert ids)
                 grouped_mlp_fwd on the local experts
                 moe_unpermute_combine with k = 1: the outputs back in received order
  exchange       all-to-all of the outputs (the reverse split sizes)
  tokens' side   moe_unpermute_combine with pos_of: out[t] = sum_j y[pos_of[t][j]]

The backward mirrors it: dout rows go out like x, the experts' side runs
grouped_mlp_bwd on the received rows (dx rows and dprob come back), and the
tokens' side combines dx and gathers dprob.  Every step is a library kernel;
the exchange is torch.distributed (NCCL between GPUs; with gloo the rows pass
through host memory).  Each expert receives its rows ordered by source rank and
then by token, which for ranks holding consecutive token ranges is the order of
the single-GPU permutation: the results equal the single-GPU layer's on the
concatenated tokens, bit for bit.

The phases are separate methods, so the exchange can also be driven by a caller
(the tests emulate several ranks in one process on one GPU that way).
"""
from __future__ import annotations

import torch

from . import binding as B

U8 = torch.uint8


class ExpertParallelFFN:
    """One rank's buffers: its T tokens over all E experts, and the rows its E/world local
    experts can receive (at most world*T*k)."""

    def __init__(self, T, H, I, E, k, world, rank, training=True, renormalize=True, device="cuda"):
        if E % world != 0:
            raise B.MoeError(2, f"world={world} must divide E={E}")
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.world, self.rank, self.training = world, rank, training
        self.El = E // world
        self.renorm = int(renormalize)
        dev = torch.device(device)
        self.dev = dev
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        z = lambda *s, dt: torch.zeros(*s, dtype=dt, device=dev)  # noqa: E731
        # tokens' side
        self.d = B.dims(T, H, I, E, k, self.renorm)
        cap = B.moe_rows_capacity(self.d)
        if cap == 0:
            raise B.MoeError(2, f"unsupported sizes T={T} H={H} I={I} E={E} k={k}")
        self.ws = z(B.moe_workspace_size(self.d, 0), dt=U8)
        self.idx = e(T, k, dt=torch.int32)
        self.prob = e(T, k, dt=torch.float32)
        self.split_sizes = e(E, dt=torch.int32)
        self.row_of = e(T, k, dt=torch.int32)
        self.src_of = e(cap, dt=torch.int32)
        self.prob_perm = e(cap, dt=torch.float32)
        self.send_x = e(T * k, H, dt=torch.bfloat16)
        self.send_prob = e(T * k, dt=torch.float32)
        self.send_eid = e(T * k, dt=torch.int32)
        self.pos_of = e(T, k, dt=torch.int32)
        self.rank_counts = e(world, dt=torch.int32)
        self.ret = e(T * k, H, dt=torch.bfloat16)          # expert outputs of this rank's rows, back
        self.out = e(T, H, dt=torch.bfloat16)
        # experts' side: the largest receive is every rank sending every row here
        self.Tr = world * T * k
        self.dl_max = B.dims(self.Tr, H, I, self.El, 1, self.renorm)
        capl = B.moe_rows_capacity(self.dl_max)
        self.capl = capl
        self.ws_l = z(B.moe_workspace_size(self.dl_max, int(training)), dt=U8)
        self.recv_x = e(self.Tr, H, dt=torch.bfloat16)
        self.recv_prob = e(self.Tr, dt=torch.float32)
        self.recv_eid = e(self.Tr, dt=torch.int32)
        self.l_split = e(self.El, dt=torch.int32)
        self.l_row_of = e(self.Tr, dt=torch.int32)
        self.l_src_of = e(capl, dt=torch.int32)
        self.l_prob_perm = e(capl, dt=torch.float32)
        self.l_xq = e(capl, H, dt=U8)
        self.l_xq_s = e(capl * H // 32, dt=U8)
        self.l_y = e(capl, H, dt=torch.bfloat16)
        self.back = e(self.Tr, H, dt=torch.bfloat16)          # outputs (or dx rows) in received order
        self.wgu_q = e(self.El, 2 * I, H, dt=U8)
        self.wgu_s = e(self.El * 2 * I * H // 32, dt=U8)
        self.wd_q = e(self.El, H, I, dt=U8)
        self.wd_s = e(self.El * H * I // 32, dt=U8)
        if training:
            self.l_xq_col = e(H, capl, dt=U8)
            self.l_xq_col_s = e(H * capl // 32, dt=U8)
            self.l_saved_gu = e(capl, 2 * I, dt=torch.bfloat16)
            self.l_aq_col = e(I, capl, dt=U8)
            self.l_aq_col_s = e(I * capl // 32, dt=U8)
            self.l_dx_perm = e(capl, H, dt=torch.bfloat16)
            self.l_dprob = e(self.Tr, 1, dt=torch.float32)
            self.dwgu = e(self.El, 2 * I, H, dt=torch.bfloat16)
            self.dwd = e(self.El, H, I, dt=torch.bfloat16)
            self.wguT_q = e(self.El, H, 2 * I, dt=U8)
            self.wguT_s = e(self.El * H * 2 * I // 32, dt=U8)
            self.wdT_q = e(self.El, I, H, dt=U8)
            self.wdT_s = e(self.El * I * H // 32, dt=U8)
            self.ret_dprob = e(T * k, dt=torch.float32)
            self.dprob = e(T, k, dt=torch.float32)
            self.dx = e(T, H, dt=torch.bfloat16)
        else:
            self.l_xq_col = self.l_xq_col_s = self.l_saved_gu = self.l_aq_col = self.l_aq_col_s = None
        self.n_recv = 0

    def dims_local(self, n_recv: int):
        return B.dims(max(n_recv, 1), self.H, self.I, self.El, 1, self.renorm)

    # ---- weights of the local experts (once per optimizer step) ----------------------
    def quantize_weights(self, w_gu_local, w_d_local, stream=None):
        """MX copies of this rank's experts' bf16 masters: [E/world][2I][H] and [E/world][H][I]."""
        El, H, I = self.El, self.H, self.I
        if self.training:
            B.mxfp8_quantize_dual(w_gu_local, El, 2 * I, H, self.wgu_q, self.wgu_s, self.wguT_q, self.wguT_s, stream)
            B.mxfp8_quantize_dual(w_d_local, El, H, I, self.wd_q, self.wd_s, self.wdT_q, self.wdT_s, stream)
        else:
            B.mxfp8_quantize(w_gu_local, El, 2 * I, H, 0, self.wgu_q, self.wgu_s, stream)
            B.mxfp8_quantize(w_d_local, El, H, I, 0, self.wd_q, self.wd_s, stream)

    # ---- phases of the forward ---------------------------------------------------------
    def dispatch_pack(self, logits, x, stream=None):
        """Route this rank's tokens and pack their rows by destination rank.  Returns
        (send_x, send_prob, send_eid, rank_counts) on the device."""
        B.moe_route(self.d, logits, self.idx, self.prob, self.split_sizes, self.row_of, self.src_of, self.prob_perm,
                    self.ws, stream)
        B.moe_ep_pack(self.d, self.world, x, self.idx, self.prob, self.row_of, self.split_sizes, self.send_x,
                      self.send_prob, self.send_eid, self.pos_of, self.rank_counts, self.ws, stream)
        return self.send_x, self.send_prob, self.send_eid, self.rank_counts

    def expert_forward(self, n_recv: int, stream=None):
        """The local experts on the n_recv rows in recv_x / recv_prob / recv_eid (already
        filled by the exchange); returns the outputs in received order (back[:n_recv])."""
        self.n_recv = n_recv
        if n_recv == 0:
            return self.back[:0]
        dl = self.dims_local(n_recv)
        B.moe_permute(dl, self.recv_eid, self.recv_prob, self.recv_x, self.l_split, self.l_row_of, self.l_src_of,
                      self.l_prob_perm, self.l_xq, self.l_xq_s, self.l_xq_col, self.l_xq_col_s, self.ws_l, stream)
        B.grouped_mlp_fwd(dl, self.l_xq, self.l_xq_s, self.l_split, self.l_prob_perm, self.wgu_q, self.wgu_s,
                          self.wd_q, self.wd_s, self.l_y, self.l_saved_gu, self.l_aq_col, self.l_aq_col_s, self.ws_l,
                          stream)
        # k = 1: the combine is a gather of every received row's output row
        B.moe_unpermute_combine(dl, self.l_y, self.l_row_of, None, self.back, stream)
        return self.back[:n_recv]

    def combine(self, stream=None):
        """out[t] = sum over j of the returned rows ret[pos_of[t][j]]."""
        B.moe_unpermute_combine(self.d, self.ret, self.pos_of, None, self.out, stream)
        return self.out

    # ---- phases of the backward -------------------------------------------------------
    def grad_pack(self, dout, stream=None):
        """dout rows packed like x (the routing of the forward)."""
        B.moe_ep_pack(self.d, self.world, dout, self.idx, self.prob, self.row_of, self.split_sizes, self.send_x,
                      self.send_prob, self.send_eid, self.pos_of, self.rank_counts, self.ws, stream)
        return self.send_x

    def expert_backward(self, stream=None):
        """The local experts' backward on the received dY rows (recv_x, the rows of the last
        expert_forward): dW of the local experts; returns the dx rows and dprob in received order."""
        n = self.n_recv
        if n == 0:
            # no rows: the local weight gradients are zero
            self.dwgu.zero_()
            self.dwd.zero_()
            return self.back[:0], self.l_dprob[:0, 0]
        dl = self.dims_local(n)
        B.grouped_mlp_bwd(dl, self.recv_x, self.l_split, self.l_row_of, self.l_src_of, self.l_prob_perm,
                          self.l_saved_gu, self.l_aq_col, self.l_aq_col_s, self.l_xq_col, self.l_xq_col_s,
                          self.wguT_q, self.wguT_s, self.wdT_q, self.wdT_s, self.l_dx_perm, self.dwgu, self.dwd,
                          self.l_dprob, self.ws_l, stream)
        B.moe_unpermute_combine(dl, self.l_dx_perm, self.l_row_of, None, self.back, stream)
        return self.back[:n], self.l_dprob[:n, 0]

    def grad_combine(self, stream=None):
        """dx[t] = sum_j of the returned dx rows ret[pos_of[t][j]]; dprob[t][j] = ret_dprob[pos_of[t][j]]."""
        B.moe_unpermute_combine(self.d, self.ret, self.pos_of, None, self.dx, stream)
        B.moe_gather_f32(self.ret_dprob, self.pos_of, self.T * self.k, self.dprob, self.ws, stream)
        return self.dx, self.dprob

    def device_error(self, stream=None):
        for ws in (self.ws, self.ws_l):
            code, site = B.moe_get_device_error(ws, stream)
            if code != 0:
                return code, site
        return 0, 0

    # ---- a whole step over a torch.distributed process group ---------------------------
    def forward(self, logits, x, group=None):
        send_x, send_prob, send_eid, counts = self.dispatch_pack(logits, x)
        in_splits, out_splits = exchange_counts(counts, group)
        n = sum(out_splits)
        all_to_all_rows(self.recv_x[:n], send_x, out_splits, in_splits, group)
        all_to_all_rows(self.recv_prob[:n], send_prob, out_splits, in_splits, group)
        all_to_all_rows(self.recv_eid[:n], send_eid, out_splits, in_splits, group)
        back = self.expert_forward(n)
        all_to_all_rows(self.ret, back, in_splits, out_splits, group)
        self._splits = (in_splits, out_splits)
        return self.combine()

    def backward(self, dout, group=None):
        in_splits, out_splits = self._splits
        n = sum(out_splits)
        send_dy = self.grad_pack(dout)
        all_to_all_rows(self.recv_x[:n], send_dy, out_splits, in_splits, group)
        back, dprob_rows = self.expert_backward()
        all_to_all_rows(self.ret, back, in_splits, out_splits, group)
        all_to_all_rows(self.ret_dprob, dprob_rows, in_splits, out_splits, group)
        return self.grad_combine()


def exchange_counts(counts, group=None):
    """All-to-all of the per-destination row counts; returns (this rank's send splits,
    its receive splits) as host lists."""
    import torch.distributed as dist
    world = counts.numel()
    backend = dist.get_backend(group)
    dev = counts.device if backend == "nccl" else torch.device("cpu")
    send = counts.to(dev, torch.int64)
    recv = torch.empty(world, dtype=torch.int64, device=dev)
    dist.all_to_all_single(recv, send, group=group)
    return send.tolist(), recv.tolist()


def all_to_all_rows(out, inp, out_splits, in_splits, group=None):
    """all_to_all_single of rows with split sizes; through host memory when the backend is gloo."""
    import torch.distributed as dist
    if dist.get_backend(group) == "nccl":
        dist.all_to_all_single(out, inp, out_splits, in_splits, group=group)
        return
    o = torch.empty(out.shape, dtype=out.dtype)
    dist.all_to_all_single(o, inp.detach().to("cpu").contiguous(), out_splits, in_splits, group=group)
    out.copy_(o)
