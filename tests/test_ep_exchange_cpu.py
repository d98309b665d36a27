"""The expert-parallel exchange (expert_routed_ffn_gemm_gb300.ep.ep_forward)
on gloo ranks on the CPU, with every compute phase done by the oracle: the
sizes, the block order of the rows and of the exponent chunks, and the path
back to the source must reproduce the oracle's whole-layer output on every
rank's tokens ("Step3.5 Flash 大模型技术深度解析" §3.2.3 / §8.1: the routed
experts spread over EP ranks, rows exchanged to their owners and back)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

E, K, D, F = 8, 2, 128, 128


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


class OracleEpBackend:
    """The three phases computed by the oracle (fp64), in the library's
    layouts: rows in dispatch order, (source, expert) blocks cut into 16-row
    exponent chunks; each chunk's exponent row is marked with (expert, chunk)
    so the source can check that the chunks come back in its own order."""

    def __init__(self, inp_bits, ep_size, ep_rank):
        self.x_unused, self.wr, self.wgu, self.wd = inp_bits
        self.ep_size, self.ep_rank = ep_size, ep_rank
        self.e_loc = E // ep_size
        self.d = D

    @staticmethod
    def _bits(rows):
        return torch.from_numpy(rows.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    def dispatch(self, x):
        import oracle

        self.x = x
        T = x.shape[0]
        xb = self._bits(x.numpy())
        idx, w, _, _ = oracle.route(xb, self.wr, K)
        counts, offsets, perm = oracle.dispatch(idx, E)
        self.idx, self.w, self.perm, self.offsets, self.T = idx, w, perm, offsets, T
        send_rows = torch.from_numpy(x.numpy()[perm // K]) if T else torch.zeros((0, D), dtype=torch.float64)
        send_w = torch.from_numpy(w.reshape(-1)[perm]) if T else torch.zeros((0,), dtype=torch.float64)
        rows = [int(offsets[(q + 1) * self.e_loc] - offsets[q * self.e_loc]) for q in range(self.ep_size)]
        return send_rows, send_w, torch.from_numpy(counts.astype(np.int32)), rows

    def experts(self, recv_rows, recv_counts, recv_w):
        import oracle

        rows = recv_rows.numpy()
        wts = recv_w.numpy()
        cnt = recv_counts.numpy().reshape(self.ep_size, self.e_loc)
        out = np.zeros_like(rows)
        exps, chunks = [], []
        pos = 0
        for s in range(self.ep_size):
            c0 = len(exps)
            for el in range(self.e_loc):
                e = self.ep_rank * self.e_loc + el
                n = int(cnt[s, el])
                if n:
                    blk = self._bits(rows[pos:pos + n])
                    out[pos:pos + n] = wts[pos:pos + n, None] * oracle.expert_ffn(blk, self.wgu, self.wd, e)
                for c in range((n + 15) // 16):
                    mark = np.zeros((D,), np.int8)
                    mark[0], mark[1] = e, c
                    exps.append(mark)
                pos += n
            chunks.append(len(exps) - c0)
        out_exp = torch.from_numpy(np.stack(exps)) if exps else torch.zeros((0, D), dtype=torch.int8)
        return torch.from_numpy(out), out_exp, chunks

    def combine(self, ret_rows, ret_exp, T):
        import oracle

        # the exponent chunks come back in this rank's own chunk order
        counts = np.diff(self.offsets[:E + 1])
        want = [(e, c) for e in range(E) for c in range((int(counts[e]) + 15) // 16)]
        got = [(int(r[0]), int(r[1])) for r in ret_exp.numpy()]
        assert got == want
        y = np.zeros((T, D))
        ret = ret_rows.numpy()
        inv = np.empty_like(self.perm)
        inv[self.perm] = np.arange(self.perm.size)
        for t in range(T):
            for j in range(K):
                y[t] += ret[inv[t * K + j]]
        if T:
            xb = self._bits(self.x.numpy())
            y += oracle.expert_ffn(xb, self.wgu, self.wd, E)
        return torch.from_numpy(y)


def _worker(rank, world, port, q):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import oracle
    from expert_routed_ffn_gemm_gb300 import ep, synth

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        shape = synth.LayerShape(T=24, d=D, E=E, k=K, F=F)
        inp = synth.make_inputs(shape, seed=5)  # every rank holds the same layer
        bits = (None, inp.w_router.numpy(), synth.bf16_bits(inp.w_gate_up), synth.bf16_bits(inp.w_down))
        T = [24, 11, 0, 17][rank]
        x = (synth.make_tokens(shape.with_tokens(T), seed=40 + rank).float().double() if T
             else torch.zeros((0, D), dtype=torch.float64))
        y = ep.ep_forward(OracleEpBackend(bits, world, rank), x, ep.dist_all_to_all())
        if T:
            xb = synth.bf16_bits(x.to(torch.bfloat16))
            ref = oracle.forward(xb, bits[1], bits[2], bits[3], K)
            np.testing.assert_allclose(y.numpy(), ref, rtol=1e-12, atol=1e-12)
        q.put((rank, T, "ok"))
    except Exception as e:  # noqa: BLE001 - reported to the parent
        q.put((rank, -1, repr(e)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_exchange_reproduces_the_whole_layer(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert all(r[2] == "ok" for r in res), "\n".join(str(r) for r in res)


def test_chunks_per_rank():
    from expert_routed_ffn_gemm_gb300 import ep

    assert ep.chunks_per_rank([17, 0, 16, 33, 1, 2], 3, 2) == [3, 5]
    assert ep.chunks_per_rank([0, 0], 1, 2) == [0, 0]
