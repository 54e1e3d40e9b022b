"""Expert parallelism over R ranks: binding of the moe_ep_* entry points and
the layer that chains them with the exchanges.

Rank r holds the E/R experts [r*E/R, (r+1)*E/R) and its own tokens. A step
(the pages deploy the layer with --enable-ep-moe --ep-size 8, "[1/2]
sgl-kernel: Fuse routed scaling factor into select_experts", sglang #8364,
Results; they do not give the exchange, read here as one all-to-all of rows
each way):

  moe_gate -> moe_ep_dispatch -> exchange counts, rows, scales ->
  moe_ep_expert_forward (local experts) -> exchange the output rows back ->
  moe_ep_combine

Every step runs in the library's kernels. The exchanges are torch.distributed
all-to-alls (NCCL between GPUs), i.e. plumbing: the binding computes only
the split sizes, from the row counts the dispatch kernel writes. The split
sizes travel to the host once per step (all_to_all_single takes them there).
"""
from . import (_check, _need_cuda, _ptr, _stream, _u8, load, moe_gate,
               moe_permute_workspace_size)


def moe_ep_dispatch(x, topk_ids, E, R, workspace=None, stream=None):
    """Pre-reorder of this rank's tokens by global expert (rank r's rows are
    the block [offsets[r*E/R], offsets[(r+1)*E/R])) plus the per-expert row
    counts. Returns (a_q, scale_a, src2dst, offsets, expert_counts)."""
    import torch
    _need_cuda(x, topk_ids, workspace)
    T, H = x.shape
    K = topk_ids.shape[1]
    dev = x.device
    M = T * K
    a_q = torch.empty((M, H), dtype=torch.uint8, device=dev)
    scale_a = torch.empty(M, dtype=torch.float32, device=dev)
    src2dst = torch.empty(M, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(moe_permute_workspace_size(T, E, K), 256),
                                dtype=torch.uint8, device=dev)
    _check("moe_ep_dispatch", load().moe_ep_dispatch(
        _ptr(x), _ptr(topk_ids), T, H, E, K, R, _ptr(a_q), _ptr(scale_a), _ptr(src2dst),
        _ptr(offsets), _ptr(counts), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return a_q, scale_a, src2dst, offsets, counts


def moe_ep_recv_reorder(recv_rows, recv_scales, recv_counts, stream=None):
    """Received rows (source blocks in rank order) -> expert-contiguous order.
    recv_counts [R, EPR] int32 on the device. Returns (a_q, scale_a, offsets,
    arrival2row)."""
    import torch
    _need_cuda(recv_rows, recv_scales, recv_counts)
    Mr, H = recv_rows.shape
    R, EPR = recv_counts.shape
    dev = recv_rows.device
    a_q = torch.empty((Mr, H), dtype=torch.uint8, device=dev)
    scale_a = torch.empty(Mr, dtype=torch.float32, device=dev)
    offsets = torch.empty(EPR + 1, dtype=torch.int32, device=dev)
    a2r = torch.empty(Mr, dtype=torch.int32, device=dev)
    ws = torch.empty(max(load().moe_ep_table_size(R, EPR), 256), dtype=torch.uint8, device=dev)
    _check("moe_ep_recv_reorder", load().moe_ep_recv_reorder(
        _ptr(_u8(recv_rows)), _ptr(recv_scales), _ptr(recv_counts), R, EPR, Mr, H, _ptr(a_q),
        _ptr(scale_a), _ptr(offsets), _ptr(a2r), _ptr(ws), ws.numel(), _stream(stream)))
    return a_q, scale_a, offsets, a2r


def moe_ep_return_gather(down, arrival2row, back=None, stream=None):
    """back[j] = down[arrival2row[j]] (bf16 rows)."""
    import torch
    _need_cuda(down, arrival2row, back)
    Mr, H = down.shape
    back = torch.empty_like(down) if back is None else back
    _check("moe_ep_return_gather", load().moe_ep_return_gather(
        _ptr(down), _ptr(arrival2row), Mr, H, _ptr(back), _stream(stream)))
    return back


def moe_ep_expert_forward(recv_rows, recv_scales, recv_counts, w13, s13, w2, s2, back=None,
                          workspace=None, stream=None):
    """The local experts on the received rows; returns the output rows
    [Mr, H] bf16 in arrival order."""
    import torch
    _need_cuda(recv_rows, recv_scales, recv_counts, w13, s13, w2, s2, back, workspace)
    Mr, H = recv_rows.shape
    R, EPR = recv_counts.shape
    I = w2.shape[2]
    if w13.shape != (EPR, 2 * I, H) or w2.shape != (EPR, H, I):
        raise ValueError("moe_ep_expert_forward: the weights must hold the EPR local experts")
    dev = recv_rows.device
    if back is None:
        back = torch.empty((Mr, H), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        nws = load().moe_ep_expert_workspace_size(Mr, H, I, R, EPR)
        workspace = torch.empty(nws, dtype=torch.uint8, device=dev)
    _check("moe_ep_expert_forward", load().moe_ep_expert_forward(
        _ptr(_u8(recv_rows)), _ptr(recv_scales), _ptr(recv_counts), R, EPR, Mr, H, I,
        _ptr(_u8(w13)), _ptr(s13), _ptr(_u8(w2)), _ptr(s2), _ptr(back), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return back


def moe_ep_combine(back_rows, src2dst, topk_w, out=None, stream=None):
    """Weighted top-k sum of the rows returned to this rank, in slot order."""
    import torch
    _need_cuda(back_rows, src2dst, topk_w, out)
    T, K = topk_w.shape
    H = back_rows.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=back_rows.device) if out is None \
        else out
    _check("moe_ep_combine", load().moe_ep_combine(
        _ptr(back_rows), _ptr(src2dst), _ptr(topk_w), T, K, H, _ptr(out), _stream(stream)))
    return out


# ---- exchanges ------------------------------------------------------------------
def split_sizes(offsets_host, recv_counts_host, R):
    """Rows this rank sends to each rank (its rows of rank r's experts) and
    receives from each rank (that rank's rows of this rank's experts)."""
    E = len(offsets_host) - 1
    EPR = E // R
    send = [int(offsets_host[(r + 1) * EPR] - offsets_host[r * EPR]) for r in range(R)]
    recv = [int(sum(recv_counts_host[s])) for s in range(R)]
    return send, recv


class DistExchange:
    """All-to-alls over a torch.distributed process group (NCCL between GPUs,
    gloo between CPU processes)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.R = dist.get_world_size(group)

    def counts(self, expert_counts):
        """Rank s sends expert_counts[r*EPR:(r+1)*EPR] to rank r; returns
        [R, EPR]: the rows each source sends for each local expert."""
        out = expert_counts.new_empty(expert_counts.shape)
        self.dist.all_to_all_single(out, expert_counts.contiguous(), group=self.group)
        return out.view(self.R, -1)

    def rows(self, t, send, recv):
        out = t.new_empty((sum(recv),) + tuple(t.shape[1:]))
        self.dist.all_to_all_single(out, t.contiguous(), output_split_sizes=list(recv),
                                    input_split_sizes=list(send), group=self.group)
        return out


class LoopbackExchange:
    """One rank holding every expert: each exchange hands the rows back to
    the same rank."""
    R = 1

    def counts(self, expert_counts):
        return expert_counts.view(1, -1).clone()

    def rows(self, t, send, recv):
        assert list(send) == list(recv)
        return t[:sum(send)].clone()


class KernelSteps:
    """The steps of an expert-parallel layer, each one of the library's entry
    points (the default of EPMoELayer)."""

    @staticmethod
    def gate(layer, logits):
        return moe_gate(logits, layer.bias, layer.num_groups, layer.topk_group, layer.top_k,
                        layer.scoring, layer.renormalize, layer.rsf)

    @staticmethod
    def dispatch(layer, x, ids):
        return moe_ep_dispatch(x, ids, layer.E, layer.R)

    @staticmethod
    def expert_forward(layer, rows, scales, recv_counts):
        return moe_ep_expert_forward(rows, scales, recv_counts, layer.w13, layer.s13, layer.w2,
                                     layer.s2)

    @staticmethod
    def combine(layer, ret, src2dst, w):
        return moe_ep_combine(ret, src2dst, w)


class EPMoELayer:
    """One rank of the expert-parallel layer: E routed experts split over
    R = exchange.R ranks, this rank holding experts [rank*E/R, (rank+1)*E/R)
    (w13 [E/R, 2I, H], w2 [E/R, H, I] and their scales). `steps` runs the
    four compute steps (KernelSteps: the library's kernels); the exchanges
    and their split sizes are this class's."""

    def __init__(self, w13, s13, w2, s2, bias, E, num_groups, topk_group, top_k, scoring,
                 renormalize, routed_scaling_factor, exchange, steps=KernelSteps):
        self.w13, self.s13, self.w2, self.s2, self.bias = w13, s13, w2, s2, bias
        self.E = E
        self.R = exchange.R
        if E % self.R != 0 or w13.shape[0] != E // self.R:
            raise ValueError("EPMoELayer: each rank holds E/R experts")
        self.num_groups, self.topk_group, self.top_k = num_groups, topk_group, top_k
        self.scoring, self.renormalize, self.rsf = scoring, renormalize, routed_scaling_factor
        self.exchange = exchange
        self.steps = steps

    def __call__(self, x, logits):
        st = self.steps
        ids, w = st.gate(self, logits)
        a_q, sa, s2d, off, cnt = st.dispatch(self, x, ids)
        recv_counts = self.exchange.counts(cnt)
        send, recv = split_sizes(off.cpu().tolist(), recv_counts.cpu().tolist(), self.R)
        rows = self.exchange.rows(a_q, send, recv)
        scales = self.exchange.rows(sa, send, recv)
        back = st.expert_forward(self, rows, scales, recv_counts)
        ret = self.exchange.rows(back, recv, send)
        return st.combine(self, ret, s2d, w)
