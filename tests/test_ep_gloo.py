"""Expert-parallel exchange on CPU ranks (gloo): the layer's split sizes,
count and row all-to-alls, receive-side merge order and return path, run by
EPMoELayer itself with the oracle standing in for the kernels. Each rank's
output must equal the oracle's whole layer on that rank's tokens (same
per-row arithmetic, so equal up to fp64 rounding), for 2 and 4 ranks.

The merge order follows the library's definition (include/moe_gb300.h,
moe_ep_recv_reorder): expert e's rows are those of source 0, then source 1,
..., each source's rows in the order it sent them."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(seed=5):
    """Global weights and tokens of a small DeepSeek-shaped layer."""
    sys.path.insert(0, ROOT)
    from moe_expert_layer_grouped_gb300 import synth
    wl = synth.Workload("ep", 96, 128, 64, 16, 4, 2, 4, synth.SIGMOID, True, 2.5, "normal")
    d = synth.make_inputs(wl, seed=seed, device="cpu")
    return wl, synth.to_numpy_inputs(d)


def recv_merge(rows, scales, recv_counts):
    """The receive-side merge (moe_ep_recv_reorder's definition), in numpy:
    returns (rows, scales, offsets, arrival2row) in expert-contiguous order."""
    R, EPR = recv_counts.shape
    Mr = rows.shape[0]
    tot = recv_counts.sum(0)
    off = np.concatenate([[0], np.cumsum(tot)]).astype(np.int32)
    a2r = np.empty(Mr, np.int32)
    j = 0
    for s in range(R):
        for e in range(EPR):
            before = int(recv_counts[:s, e].sum())
            for i in range(int(recv_counts[s, e])):
                a2r[j] = off[e] + before + i
                j += 1
    assert j == Mr
    out_rows = np.empty_like(rows)
    out_scales = np.empty_like(scales)
    out_rows[a2r] = rows
    out_scales[a2r] = scales
    return out_rows, out_scales, off, a2r


class OracleSteps:
    """EPMoELayer's compute steps done by the oracle on CPU tensors."""

    @staticmethod
    def gate(layer, logits):
        import torch
        import oracle
        ids, w = oracle.gate(logits.numpy(), None if layer.bias is None else layer.bias.numpy(),
                             layer.num_groups, layer.topk_group, layer.top_k, layer.scoring,
                             layer.renormalize, layer.rsf)
        return torch.from_numpy(ids), torch.from_numpy(w)

    @staticmethod
    def dispatch(layer, x, ids):
        import torch
        import oracle
        a_q, sa, s2d, off = oracle.permute_quant(x.numpy(), ids.numpy(), layer.E)
        cnt = np.diff(off).astype(np.int32)
        return (torch.from_numpy(a_q), torch.from_numpy(sa), torch.from_numpy(s2d),
                torch.from_numpy(off), torch.from_numpy(cnt))

    @staticmethod
    def expert_forward(layer, rows, scales, recv_counts):
        import torch
        import oracle
        a_q, sa, off, a2r = recv_merge(rows.numpy(), scales.numpy(), recv_counts.numpy())
        h = oracle.silu_mul(oracle.grouped_gemm(a_q, sa, layer.w13.numpy(), layer.s13.numpy(),
                                                off))
        q2, sa2 = oracle.act_quant(oracle.bf16_round(h))
        down = oracle.grouped_gemm(q2, sa2, layer.w2.numpy(), layer.s2.numpy(), off)
        return torch.from_numpy(down[a2r])

    @staticmethod
    def combine(layer, ret, src2dst, w):
        import oracle
        return oracle.unpermute_sum(ret.numpy(), src2dst.numpy(), w.numpy())


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    from moe_expert_layer_grouped_gb300 import ep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl, n = _problem()
        E, EPR = wl.E, wl.E // world
        lo, hi = rank * EPR, (rank + 1) * EPR
        T_r = wl.T // world
        tok = slice(rank * T_r, (rank + 1) * T_r)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
        layer = ep.EPMoELayer(t(n["w13"][lo:hi]), t(n["s13"][lo:hi]), t(n["w2"][lo:hi]),
                              t(n["s2"][lo:hi]), t(n["bias"]), E, wl.num_groups,
                              wl.topk_group, wl.top_k, wl.scoring, wl.renormalize, wl.rsf,
                              ep.DistExchange(), steps=OracleSteps)
        out = layer(t(n["x"][tok]), t(n["logits"][tok]))
        ref, _, _ = oracle.forward_tokens(n["x"], n["logits"], n["bias"], n["w13"], n["s13"],
                                          n["w2"], n["s2"], wl.num_groups, wl.topk_group,
                                          wl.top_k, wl.scoring, wl.renormalize, wl.rsf,
                                          tokens=np.arange(wl.T)[tok])
        err = float(np.abs(out - ref).max() / np.abs(ref).max())
        # this rank's received rows: every slot of every rank routed to its experts
        ids, _ = oracle.gate(n["logits"], n["bias"], wl.num_groups, wl.topk_group, wl.top_k,
                             wl.scoring, wl.renormalize, wl.rsf)
        mine = int(((ids >= lo) & (ids < hi)).sum())
        dist.barrier()
        q.put((rank, err, mine))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_ep_layer_over_gloo_ranks_matches_the_oracle(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err, mine in res:
        assert err <= 1e-12, (rank, err)
    assert len(res) == world


def test_split_sizes_and_merge_order():
    from moe_expert_layer_grouped_gb300 import ep
    # rank 1 of 2, 3 experts each: its offsets over 6 global experts
    off = [0, 2, 2, 5, 6, 9, 9]
    recv_counts = [[1, 0, 2], [0, 3, 1]]       # from ranks 0 and 1, its experts 3..5
    send, recv = ep.split_sizes(off, recv_counts, 2)
    assert send == [5, 4] and recv == [3, 4]
    rows = np.arange(7, dtype=np.uint8).reshape(7, 1)
    sc = np.arange(7, dtype=np.float32)
    out, osc, o, a2r = recv_merge(rows, sc, np.array(recv_counts, np.int32))
    assert o.tolist() == [0, 1, 4, 7]
    # expert 0: src0's row 0; expert 1: src1's rows 3,4,5; expert 2: src0's rows 1,2 then src1's 6
    assert out[:, 0].tolist() == [0, 3, 4, 5, 1, 2, 6]
    assert a2r.tolist() == [0, 4, 5, 1, 2, 3, 6]
    assert np.array_equal(osc[a2r], sc)
