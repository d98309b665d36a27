"""Expert-parallel layer calls over several ranks.

"Step3.5 Flash 大模型技术深度解析" (jsqmd.com) §3.2.3 and §8.1 place the 288
routed experts on 8 GPUs (36 each) and move every token row to the GPU that
owns its expert and back.  Here rank r of ``ep_size`` owns the routed experts
[r*E_loc, (r+1)*E_loc) and a copy of the shared expert; one layer call is the
library's three phases (``moe_ep_dispatch``, ``moe_ep_experts``,
``moe_ep_combine`` in include/moe.h) around two all-to-all exchanges:

1. dispatch: route this rank's tokens, lay the routed rows out expert by
   expert; rank q's rows are one block;
2. exchange the per-expert counts, the rows and their gate weights;
3. experts: run the local experts over the received (source, expert) blocks;
4. exchange the output rows and their exponent chunks back to their sources;
5. combine: the shared expert on this rank's tokens and the fixed-order sum.

This module only moves tensors and sizes; every step of the arithmetic runs in
the library's kernels (``GpuEpBackend``).  ``ep_forward`` takes the exchange as
a function, so the same code runs over ``torch.distributed``
(``dist_all_to_all``) or over ranks simulated as threads of one process
(``LocalExchange``).
"""
from __future__ import annotations

import threading

import torch

from . import binding

Y_ROWS_PER_CHUNK = 16  # rows per exponent chunk of the scaled fp16 expert outputs


def chunks_per_rank(counts: list[int], e_loc: int, ep_size: int) -> list[int]:
    """Exponent chunks of the rows a source sends to each rank: every expert's
    rows are cut into 16-row chunks from the expert's first row."""
    return [sum((c + Y_ROWS_PER_CHUNK - 1) // Y_ROWS_PER_CHUNK for c in counts[q * e_loc:(q + 1) * e_loc])
            for q in range(ep_size)]


class GpuEpBackend:
    """One rank's library handle for the three phases (bf16 weights: the router
    over all E experts, this rank's experts then the shared expert)."""

    def __init__(self, w_router, w_gate_up_local, w_down_local, top_k: int, max_tokens: int, ep_size: int,
                 ep_rank: int, max_recv_rows: int, has_shared: bool = True, out_fp32: bool = False):
        E, d = w_router.shape
        G, twoF, _ = w_gate_up_local.shape
        self.F = twoF // 2
        self.d, self.E, self.k = d, E, top_k
        self.ep_size, self.ep_rank = ep_size, ep_rank
        self.e_loc = E // ep_size
        if G != self.e_loc + int(has_shared):
            raise ValueError("local weights must hold E/ep_size experts (+ the shared expert)")
        self.out_fp32 = out_fp32
        self.device = w_gate_up_local.device
        self.weights = (w_router, w_gate_up_local, w_down_local)  # borrowed by the handle
        layer = binding.moe_config(d, E, top_k, self.F, int(has_shared), max_tokens, int(out_fp32))
        cfg = binding.moe_ep_config(layer, ep_size, ep_rank, max_recv_rows)
        self.handle = binding.moe_ep_init(cfg, w_router, w_gate_up_local, w_down_local)

    def dispatch(self, x: torch.Tensor):
        T = x.shape[0]
        send_rows = torch.empty((T * self.k, self.d), dtype=torch.bfloat16, device=self.device)
        send_w = torch.empty((T * self.k,), dtype=torch.float32, device=self.device)
        send_counts = torch.empty((self.E,), dtype=torch.int32, device=self.device)
        rows = binding.moe_ep_dispatch(self.handle, x, T, send_rows, send_w, send_counts, self.ep_size)
        return send_rows, send_w, send_counts, rows

    def experts(self, recv_rows, recv_counts, recv_w):
        n = recv_rows.shape[0]
        max_chunks = n // Y_ROWS_PER_CHUNK + self.ep_size * self.e_loc
        out_rows = torch.empty((n, self.d), dtype=torch.float16, device=self.device)
        out_exp = torch.empty((max_chunks, self.d), dtype=torch.int8, device=self.device)
        chunks = binding.moe_ep_experts(self.handle, recv_rows, recv_counts, recv_w, n, out_rows, out_exp,
                                        self.ep_size)
        return out_rows, out_exp[:sum(chunks)], chunks

    def combine(self, ret_rows, ret_exp, T: int):
        y = torch.empty((T, self.d), dtype=torch.float32 if self.out_fp32 else torch.bfloat16, device=self.device)
        binding.moe_ep_combine(self.handle, ret_rows, ret_exp, y)
        return y

    def close(self):
        if getattr(self, "handle", None):
            binding.moe_free(self.handle)
            self.handle = None


def dist_all_to_all(group=None):
    """The exchange over torch.distributed (NCCL for device tensors)."""
    import torch.distributed as dist

    def a2a(inp: torch.Tensor, out_splits: list[int], in_splits: list[int]) -> torch.Tensor:
        out = inp.new_empty((sum(out_splits),) + tuple(inp.shape[1:]))
        dist.all_to_all_single(out, inp.contiguous(), output_split_sizes=out_splits, input_split_sizes=in_splits,
                               group=group)
        return out

    return a2a


class LocalExchange:
    """All-to-all among ranks run as threads of one process (each thread calls
    ``for_rank(r)``'s function the same number of times, in the same order)."""

    def __init__(self, n: int):
        self.n = n
        self.barrier = threading.Barrier(n)
        self.box = [[None] * n for _ in range(n)]

    def for_rank(self, r: int):
        def a2a(inp: torch.Tensor, out_splits: list[int], in_splits: list[int]) -> torch.Tensor:
            parts = torch.split(inp, in_splits)
            for q in range(self.n):
                self.box[r][q] = parts[q]
            self.barrier.wait()
            out = torch.cat([self.box[q][r] for q in range(self.n)])
            if out.shape[0] != sum(out_splits):
                raise RuntimeError("exchange sizes disagree between ranks")
            self.barrier.wait()
            return out

        return a2a


def ep_forward(backend, x: torch.Tensor, a2a) -> torch.Tensor:
    """One expert-parallel layer call of this rank's tokens x [T, d]."""
    S, e_loc = backend.ep_size, backend.e_loc
    send_rows, send_w, send_counts, rows_per_rank = backend.dispatch(x)
    # counts: rank q gets the [E_loc] slice of every source, in source order
    recv_counts = a2a(send_counts.view(S, e_loc), [1] * S, [1] * S).contiguous()
    recv_per_src = [int(v) for v in recv_counts.sum(dim=1).tolist()]
    recv_rows = a2a(send_rows, recv_per_src, rows_per_rank)
    recv_w = a2a(send_w, recv_per_src, rows_per_rank)
    out_rows, out_exp, chunks_per_src = backend.experts(recv_rows, recv_counts.view(-1), recv_w)
    # back to the sources: the blocks come back in rank order, which is this
    # rank's own dispatch order (rows and exponent chunks alike)
    my_chunks = chunks_per_rank([int(v) for v in send_counts.tolist()], e_loc, S)
    ret_rows = a2a(out_rows, rows_per_rank, recv_per_src)
    ret_exp = a2a(out_exp, my_chunks, chunks_per_src)
    return backend.combine(ret_rows, ret_exp, x.shape[0])
