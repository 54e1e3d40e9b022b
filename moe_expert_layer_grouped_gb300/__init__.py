"""Python binding of libmoe_gb300.so, the C ABI of the grouped-expert MoE
layer forward on GB300 (sm_103a).

The functions carry the C entry points' names and only marshal arguments:
they allocate output tensors with torch when none are given, pass raw device
pointers, sizes and the current CUDA stream, and raise MoEError on a
non-zero status. Every step of the layer runs in the library's CUDA kernels;
there is no fallback: if the library is not built, every call raises.

Tensor formats: bf16 tensors are torch.bfloat16; FP8 e4m3 tensors are
torch.uint8 (codes) or torch.float8_e4m3fn; everything is contiguous and on
the same CUDA device.
"""
import ctypes
import os

__all__ = [
    "MoEError", "SIGMOID", "SOFTMAX", "EPI_BF16", "EPI_SILU_MUL", "library_path", "load",
    "moe_gate", "moe_permute_quant", "moe_permute_workspace_size", "moe_grouped_gemm",
    "moe_forward_shared", "moe_forward_shared_host", "moe_permute_quant_block",
    "moe_grouped_gemm_block", "moe_act_quant_block", "moe_block_workspace_size",
    "moe_forward_block", "moe_forward_block_host", "moe_test_gemm_timeout",
    "moe_permute_quant_noalloc", "moe_permute_quant_rows", "moe_grouped_gemm_rows",
    "moe_permute_quant_nvfp4", "moe_act_quant_nvfp4", "moe_grouped_gemm_nvfp4",
    "moe_nvfp4_workspace_size", "moe_forward_nvfp4", "moe_forward_nvfp4_host",
    "moe_nvfp4_arrange_scales", "moe_test_gemm_nvfp4_timeout",
    "moe_act_quant", "moe_unpermute_sum", "moe_workspace_size", "moe_forward",
    "moe_forward_host", "moe_device_status", "MoELayer", "QUANT_TOKEN", "QUANT_BLOCK",
    "QUANT_NVFP4", "MoELayerDesc", "moe_pipeline_workspace_size", "moe_forward_host_pipelined",
    # expert parallelism (moe_expert_layer_grouped_gb300.ep)
    "moe_ep_dispatch", "moe_ep_recv_reorder", "moe_ep_return_gather", "moe_ep_expert_forward",
    "moe_ep_combine", "EPMoELayer",
]

SIGMOID = 0
SOFTMAX = 1
EPI_BF16 = 0
EPI_SILU_MUL = 1
QUANT_TOKEN = 0
QUANT_BLOCK = 1
QUANT_NVFP4 = 2
# device error codes read by moe_device_status()
DEV_OK = 0
DEV_BAD_EXPERT_ID = 1
DEV_PIPE_TIMEOUT = 2
DEV_BAD_OFFSETS = 3

_STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
           -3: "MOE_ERR_WORKSPACE", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE"}

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path():
    return os.path.join(_HERE, "_lib", "libmoe_gb300.so")


class MoEError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {_STATUS.get(status, status)}")


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t


class MoELayerDesc(ctypes.Structure):
    """struct moe_layer of the C header: the layer a pipelined call runs."""
    _fields_ = [("quant", _I), ("T", _I), ("H", _I), ("I", _I), ("E", _I), ("n_shared", _I),
                ("num_groups", _I), ("topk_group", _I), ("top_k", _I), ("scoring", _I),
                ("renormalize", _I), ("routed_scaling_factor", _F), ("bias", _P),
                ("w13", _P), ("s13", _P), ("w2", _P), ("s2", _P), ("g13", _P), ("g2", _P),
                ("ga1", _F), ("ga2", _F)]


_SIGNATURES = {
    "moe_pipeline_workspace_size": (_SZ, [ctypes.POINTER(MoELayerDesc)]),
    "moe_forward_host_pipelined": (_I, [ctypes.POINTER(MoELayerDesc), _I, _P, _P, _P, _P, _SZ,
                                        _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_abi_version": (_I, []),
    "moe_gate": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "moe_permute_workspace_size": (_SZ, [_I, _I, _I]),
    "moe_permute_quant": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_quant_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_grouped_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_act_quant": (_I, [_P, _P, _I, _I, _P, _P, _P]),
    "moe_unpermute_sum": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                         _P, _P, _SZ, _P]),
    "moe_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                              _F, _P, _P, _SZ, _P]),
    "moe_forward_shared": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                _I, _F, _P, _P, _SZ, _P]),
    "moe_forward_shared_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                     _I, _I, _F, _P, _P, _SZ, _P]),
    "moe_permute_quant_block": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_gemm_block": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_act_quant_block": (_I, [_P, _I, _I, _P, _P, _P]),
    "moe_block_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_test_gemm_timeout": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _P]),
    "moe_forward_block": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                               _I, _F, _P, _P, _SZ, _P]),
    "moe_forward_block_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                    _I, _I, _F, _P, _P, _SZ, _P]),
    "moe_device_status": (_I, [ctypes.POINTER(_I)]),
    "moe_permute_quant_rows": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_gemm_rows": (_I, [_P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_permute_quant_nvfp4": (_I, [_P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_act_quant_nvfp4": (_I, [_P, _I, _I, _F, _P, _P, _P]),
    "moe_grouped_gemm_nvfp4": (_I, [_P, _P, _F, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_test_gemm_nvfp4_timeout": (_I, [_P, _P, _F, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I,
                                         _P]),
    "moe_nvfp4_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_nvfp4_arrange_scales": (_I, [_P, _I, _I, _I, _I, _P, _P]),
    "moe_forward_nvfp4": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _F, _I, _I, _I, _I, _I,
                               _I, _I, _I, _I, _I, _F, _P, _P, _SZ, _P]),
    "moe_forward_nvfp4_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _F, _I, _I, _I, _I,
                                    _I, _I, _I, _I, _I, _I, _F, _P, _P, _SZ, _P]),
    "moe_ep_table_size": (_SZ, [_I, _I]),
    "moe_ep_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_ep_recv_reorder": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_ep_return_gather": (_I, [_P, _P, _I, _I, _P, _P]),
    "moe_ep_expert_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_ep_expert_forward": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ,
                                   _P]),
    "moe_ep_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
}


def load():
    """Load libmoe_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; "
                f"g.build()'` (needs nvcc); the MoE layer has no non-CUDA path")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(fn, status):
    if status != 0:
        raise MoEError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("moe_gb300: tensors must be CUDA tensors")
            if not t.is_contiguous():
                raise ValueError("moe_gb300: tensors must be contiguous")


def _need_buf(fn, name, t, numel, dtypes):
    """A caller-supplied output buffer must hold `numel` elements of one of
    `dtypes`: a smaller one would be written past its end by the kernels."""
    if t.numel() != numel or t.dtype not in dtypes:
        raise ValueError(f"{fn}: {name} must hold {numel} elements of "
                         f"{' or '.join(str(d) for d in dtypes)}, got {t.numel()} of {t.dtype}")


def _gemm_bufs(fn, M, N, E, cols, scale_a, n_sa, scale_b, n_sb, offsets, C, row_amax,
               scale_dtypes=None):
    """The grouped GEMM's scale, offset and output tensors must hold what the
    kernels read and write (an undersized one would be read or written past
    its end on the device)."""
    import torch
    sd = scale_dtypes or (torch.float32,)
    _need_buf(fn, "scale_a", scale_a, n_sa, sd)
    _need_buf(fn, "scale_b", scale_b, n_sb, sd)
    _need_buf(fn, "offsets", offsets, E + 1, (torch.int32,))
    _need_buf(fn, "C", C, M * cols, (torch.bfloat16,))
    if row_amax is not None:
        _need_buf(fn, "row_amax", row_amax, M, (torch.float32,))


def _permute_bufs(fn, T, H, K, E, a_q, scale_a, src2dst, offsets, scales_per_row=1):
    import torch
    M = T * K
    if a_q is not None:
        _need_buf(fn, "a_q", a_q, M * H, (torch.uint8, torch.float8_e4m3fn))
    if scale_a is not None:
        _need_buf(fn, "scale_a", scale_a, M * scales_per_row, (torch.float32,))
    if src2dst is not None:
        _need_buf(fn, "src2dst", src2dst, M, (torch.int32,))
    if offsets is not None:
        _need_buf(fn, "offsets", offsets, E + 1, (torch.int32,))


def _u8(t):
    import torch
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


def moe_gate(logits, bias, num_groups, topk_group, top_k, scoring=SIGMOID, renormalize=True,
             routed_scaling_factor=1.0, topk_ids=None, topk_w=None, stream=None):
    import torch
    _need_cuda(logits, bias)
    T, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _check("moe_gate", load().moe_gate(
        _ptr(logits), _ptr(bias), T, E, num_groups, topk_group, top_k, scoring,
        int(bool(renormalize)), float(routed_scaling_factor), _ptr(topk_ids), _ptr(topk_w),
        _stream(stream)))
    return topk_ids, topk_w


def moe_permute_workspace_size(T, E, K):
    return load().moe_permute_workspace_size(T, E, K)


def moe_permute_quant(x, topk_ids, E, a_q=None, scale_a=None, src2dst=None, offsets=None,
                      workspace=None, stream=None):
    import torch
    _need_cuda(x, topk_ids, a_q, scale_a, src2dst, offsets)
    T, H = x.shape
    K = topk_ids.shape[1]
    _permute_bufs("moe_permute_quant", T, H, K, E, a_q, scale_a, src2dst, offsets)
    dev = x.device
    M = T * K
    a_q = torch.empty((M, H), dtype=torch.uint8, device=dev) if a_q is None else a_q
    scale_a = torch.empty(M, dtype=torch.float32, device=dev) if scale_a is None else scale_a
    src2dst = torch.empty(M, dtype=torch.int32, device=dev) if src2dst is None else src2dst
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    nws = moe_permute_workspace_size(T, E, K)
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
    _check("moe_permute_quant", load().moe_permute_quant(
        _ptr(x), _ptr(topk_ids), T, H, E, K, _ptr(_u8(a_q)), _ptr(scale_a), _ptr(src2dst),
        _ptr(offsets), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return a_q, scale_a, src2dst, offsets


def moe_permute_quant_noalloc(x, topk_ids, E, a_q, scale_a, src2dst, offsets, stream=None):
    """moe_permute_quant for callers that cannot allocate: the caller passes
    every output buffer and the library uses its fixed device scratch instead
    of a workspace (see include/moe_gb300.h for the size limit and the rule
    that overlapping calls race). Allocates nothing."""
    _need_cuda(x, topk_ids, a_q, scale_a, src2dst, offsets)
    T, H = x.shape
    K = topk_ids.shape[1]
    _permute_bufs("moe_permute_quant_noalloc", T, H, K, E, a_q, scale_a, src2dst, offsets)
    _check("moe_permute_quant_noalloc", load().moe_permute_quant_noalloc(
        _ptr(x), _ptr(topk_ids), T, H, E, K, _ptr(_u8(a_q)), _ptr(scale_a), _ptr(src2dst),
        _ptr(offsets), _stream(stream)))
    return a_q, scale_a, src2dst, offsets


def moe_permute_quant_rows(x, topk_ids, E, workspace=None, stream=None):
    """Pre-reorder storing each token's codes once, in token order. Returns
    (a_tok [T,H], scale_a [T*K], src2dst [T*K], row_token [T*K], offsets)."""
    import torch
    _need_cuda(x, topk_ids, workspace)
    T, H = x.shape
    K = topk_ids.shape[1]
    dev = x.device
    M = T * K
    a_tok = torch.empty((T, H), dtype=torch.uint8, device=dev)
    scale_a = torch.empty(M, dtype=torch.float32, device=dev)
    src2dst = torch.empty(M, dtype=torch.int32, device=dev)
    row_token = torch.empty(M, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(moe_permute_workspace_size(T, E, K), 256), dtype=torch.uint8,
                                device=dev)
    _check("moe_permute_quant_rows", load().moe_permute_quant_rows(
        _ptr(x), _ptr(topk_ids), T, H, E, K, _ptr(a_tok), _ptr(scale_a), _ptr(src2dst),
        _ptr(row_token), _ptr(offsets), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return a_tok, scale_a, src2dst, row_token, offsets


def moe_grouped_gemm_rows(A_tok, row_token, scale_a, B, scale_b, offsets, epilogue=EPI_BF16,
                          C=None, row_amax=None, stream=None):
    """moe_grouped_gemm with permuted row r of A = A_tok[row_token[r]]."""
    import torch
    _need_cuda(A_tok, row_token, scale_a, B, scale_b, offsets, C, row_amax)
    T, Kd = A_tok.shape
    M = row_token.numel()
    E, N, Kd2 = B.shape
    if Kd != Kd2:
        raise ValueError("moe_grouped_gemm_rows: K mismatch")
    cols = N // 2 if epilogue == EPI_SILU_MUL else N
    if C is None:
        C = torch.empty((M, cols), dtype=torch.bfloat16, device=A_tok.device)
    _gemm_bufs("moe_grouped_gemm_rows", M, N, E, cols, scale_a, M, scale_b, E * N, offsets, C,
               row_amax)
    _check("moe_grouped_gemm_rows", load().moe_grouped_gemm_rows(
        _ptr(_u8(A_tok)), T, _ptr(row_token), _ptr(scale_a), _ptr(_u8(B)), _ptr(scale_b),
        _ptr(offsets), M, N, Kd, E, epilogue, _ptr(C), _ptr(row_amax), _stream(stream)))
    return C


def moe_grouped_gemm(A, scale_a, B, scale_b, offsets, epilogue=EPI_BF16, C=None, row_amax=None,
                     stream=None):
    import torch
    _need_cuda(A, scale_a, B, scale_b, offsets, C, row_amax)
    M, Kd = A.shape
    E, N, Kd2 = B.shape
    if Kd2 != Kd:
        raise ValueError("moe_grouped_gemm: K mismatch")
    cols = N // 2 if epilogue == EPI_SILU_MUL else N
    if C is None:
        C = torch.empty((M, cols), dtype=torch.bfloat16, device=A.device)
    _gemm_bufs("moe_grouped_gemm", M, N, E, cols, scale_a, M, scale_b, E * N, offsets, C,
               row_amax)
    _check("moe_grouped_gemm", load().moe_grouped_gemm(
        _ptr(_u8(A)), _ptr(scale_a), _ptr(_u8(B)), _ptr(scale_b), _ptr(offsets), M, N, Kd, E,
        epilogue, _ptr(C), _ptr(row_amax), _stream(stream)))
    return C


def moe_act_quant(h, row_amax=None, q=None, scale=None, stream=None):
    import torch
    _need_cuda(h, row_amax)
    M, I = h.shape
    q = torch.empty((M, I), dtype=torch.uint8, device=h.device) if q is None else q
    scale = torch.empty(M, dtype=torch.float32, device=h.device) if scale is None else scale
    _need_cuda(q, scale)
    _need_buf("moe_act_quant", "q", q, M * I, (torch.uint8, torch.float8_e4m3fn))
    _need_buf("moe_act_quant", "scale", scale, M, (torch.float32,))
    if row_amax is not None:
        _need_buf("moe_act_quant", "row_amax", row_amax, M, (torch.float32,))
    _check("moe_act_quant", load().moe_act_quant(
        _ptr(h), _ptr(row_amax), M, I, _ptr(_u8(q)), _ptr(scale), _stream(stream)))
    return q, scale


def moe_unpermute_sum(down, src2dst, topk_w, out=None, stream=None):
    import torch
    _need_cuda(down, src2dst, topk_w)
    T, K = topk_w.shape
    H = down.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=down.device) if out is None else out
    _need_cuda(out)
    _need_buf("moe_unpermute_sum", "down", down, T * K * H, (torch.bfloat16,))
    _need_buf("moe_unpermute_sum", "src2dst", src2dst, T * K, (torch.int32,))
    _need_buf("moe_unpermute_sum", "topk_w", topk_w, T * K, (torch.float32,))
    _need_buf("moe_unpermute_sum", "out", out, T * H, (torch.bfloat16,))
    _check("moe_unpermute_sum", load().moe_unpermute_sum(
        _ptr(down), _ptr(src2dst), _ptr(topk_w), T, K, H, _ptr(out), _stream(stream)))
    return out


def moe_workspace_size(T, H, I, E, K):
    return load().moe_workspace_size(T, H, I, E, K)


def _dims(x, logits, w13, w2, n_shared=0):
    T, H = x.shape
    E = logits.shape[1]
    I = w2.shape[2]
    n = E + n_shared
    if tuple(w13.shape) != (n, 2 * I, H) or tuple(w2.shape) != (n, H, I):
        raise ValueError("moe_forward: weight shapes do not match [E+n_shared,2I,H] / "
                         "[E+n_shared,H,I]")
    return T, H, I, E


def moe_forward(x, logits, bias, w13, s13, w2, s2, num_groups, topk_group, top_k,
                scoring=SIGMOID, renormalize=True, routed_scaling_factor=1.0, out=None,
                workspace=None, stream=None):
    import torch
    _need_cuda(x, logits, bias, w13, s13, w2, s2, out, workspace)
    T, H, I, E = _dims(x, logits, w13, w2)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device) if out is None else out
    _need_buf("moe_forward", "out", out, T * H, (torch.bfloat16,))
    nws = moe_workspace_size(T, H, I, E, top_k)
    if workspace is None:
        workspace = torch.empty(nws, dtype=torch.uint8, device=x.device)
    _check("moe_forward", load().moe_forward(
        _ptr(x), _ptr(logits), _ptr(bias), _ptr(_u8(w13)), _ptr(s13), _ptr(_u8(w2)), _ptr(s2),
        T, H, I, E, num_groups, topk_group, top_k, scoring, int(bool(renormalize)),
        float(routed_scaling_factor), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def moe_forward_host(x_host, logits_host, bias, w13, s13, w2, s2, num_groups, topk_group, top_k,
                     scoring, renormalize, routed_scaling_factor, out_host, workspace,
                     stream=None):
    """x_host, logits_host and out_host are CPU tensors (pinned for asynchrony);
    the copies run on `stream` inside the call."""
    _need_cuda(bias, w13, s13, w2, s2, workspace)
    for t in (x_host, logits_host, out_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("moe_forward_host: x, logits and out must be contiguous host tensors")
    T, H, I, E = _dims(x_host, logits_host, w13, w2)
    _check("moe_forward_host", load().moe_forward_host(
        _ptr(x_host), _ptr(logits_host), _ptr(bias), _ptr(_u8(w13)), _ptr(s13), _ptr(_u8(w2)),
        _ptr(s2), T, H, I, E, num_groups, topk_group, top_k, scoring, int(bool(renormalize)),
        float(routed_scaling_factor), _ptr(out_host), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out_host


def moe_forward_shared(x, logits, bias, w13, s13, w2, s2, n_shared, num_groups, topk_group,
                       top_k, scoring=SIGMOID, renormalize=True, routed_scaling_factor=1.0,
                       out=None, workspace=None, stream=None):
    """moe_forward plus n_shared shared experts stored as experts E.. of w13/w2."""
    import torch
    _need_cuda(x, logits, bias, w13, s13, w2, s2, out, workspace)
    T, H, I, E = _dims(x, logits, w13, w2, n_shared)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device) if out is None else out
    _need_buf("moe_forward_shared", "out", out, T * H, (torch.bfloat16,))
    if workspace is None:
        nws = moe_workspace_size(T, H, I, E + n_shared, top_k + n_shared)
        workspace = torch.empty(nws, dtype=torch.uint8, device=x.device)
    _check("moe_forward_shared", load().moe_forward_shared(
        _ptr(x), _ptr(logits), _ptr(bias), _ptr(_u8(w13)), _ptr(s13), _ptr(_u8(w2)), _ptr(s2),
        T, H, I, E, int(n_shared), num_groups, topk_group, top_k, scoring,
        int(bool(renormalize)), float(routed_scaling_factor), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def moe_forward_shared_host(x_host, logits_host, bias, w13, s13, w2, s2, n_shared, num_groups,
                            topk_group, top_k, scoring, renormalize, routed_scaling_factor,
                            out_host, workspace, stream=None):
    """moe_forward_shared with x, logits and out in host memory (as moe_forward_host)."""
    _need_cuda(bias, w13, s13, w2, s2, workspace)
    for t in (x_host, logits_host, out_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("moe_forward_shared_host: x, logits and out must be contiguous "
                             "host tensors")
    T, H, I, E = _dims(x_host, logits_host, w13, w2, n_shared)
    _check("moe_forward_shared_host", load().moe_forward_shared_host(
        _ptr(x_host), _ptr(logits_host), _ptr(bias), _ptr(_u8(w13)), _ptr(s13), _ptr(_u8(w2)),
        _ptr(s2), T, H, I, E, int(n_shared), num_groups, topk_group, top_k, scoring,
        int(bool(renormalize)), float(routed_scaling_factor), _ptr(out_host), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out_host


# ---- block-quantised FP8 (128-channel activation scales, 128 x 128 weight scales)
def moe_permute_quant_block(x, topk_ids, E, a_q=None, scale_a=None, src2dst=None, offsets=None,
                            workspace=None, stream=None):
    """moe_permute_quant with one scale per token per 128 channels: scale_a [T*K, H/128]."""
    import torch
    _need_cuda(x, topk_ids, a_q, scale_a, src2dst, offsets)
    T, H = x.shape
    K = topk_ids.shape[1]
    _permute_bufs("moe_permute_quant_block", T, H, K, E, a_q, scale_a, src2dst, offsets,
                  scales_per_row=H // 128)
    dev = x.device
    M = T * K
    a_q = torch.empty((M, H), dtype=torch.uint8, device=dev) if a_q is None else a_q
    if scale_a is None:
        scale_a = torch.empty((M, H // 128), dtype=torch.float32, device=dev)
    src2dst = torch.empty(M, dtype=torch.int32, device=dev) if src2dst is None else src2dst
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    if workspace is None:
        workspace = torch.empty(max(moe_permute_workspace_size(T, E, K), 256), dtype=torch.uint8,
                                device=dev)
    _check("moe_permute_quant_block", load().moe_permute_quant_block(
        _ptr(x), _ptr(topk_ids), T, H, E, K, _ptr(_u8(a_q)), _ptr(scale_a), _ptr(src2dst),
        _ptr(offsets), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return a_q, scale_a, src2dst, offsets


def moe_grouped_gemm_block(A, scale_a, B, scale_b, offsets, epilogue=EPI_BF16, C=None,
                           stream=None):
    """scale_a [M, Kd/128]; scale_b [E, N/128, Kd/128]."""
    import torch
    _need_cuda(A, scale_a, B, scale_b, offsets, C)
    M, Kd = A.shape
    E, N, Kd2 = B.shape
    if Kd2 != Kd:
        raise ValueError("moe_grouped_gemm_block: K mismatch")
    cols = N // 2 if epilogue == EPI_SILU_MUL else N
    if C is None:
        C = torch.empty((M, cols), dtype=torch.bfloat16, device=A.device)
    _gemm_bufs("moe_grouped_gemm_block", M, N, E, cols, scale_a, M * (Kd // 128), scale_b,
               E * (N // 128) * (Kd // 128), offsets, C, None)
    _check("moe_grouped_gemm_block", load().moe_grouped_gemm_block(
        _ptr(_u8(A)), _ptr(scale_a), _ptr(_u8(B)), _ptr(scale_b), _ptr(offsets), M, N, Kd, E,
        epilogue, _ptr(C), _stream(stream)))
    return C


def moe_act_quant_block(h, q=None, scale=None, stream=None):
    """Requantisation with one scale per row per 128 channels: scale [M, I/128]."""
    import torch
    _need_cuda(h)
    M, I = h.shape
    q = torch.empty((M, I), dtype=torch.uint8, device=h.device) if q is None else q
    if scale is None:
        scale = torch.empty((M, I // 128), dtype=torch.float32, device=h.device)
    _need_cuda(q, scale)
    _need_buf("moe_act_quant_block", "q", q, M * I, (torch.uint8, torch.float8_e4m3fn))
    _need_buf("moe_act_quant_block", "scale", scale, M * (I // 128), (torch.float32,))
    _check("moe_act_quant_block", load().moe_act_quant_block(
        _ptr(h), M, I, _ptr(_u8(q)), _ptr(scale), _stream(stream)))
    return q, scale


def moe_block_workspace_size(T, H, I, E, K):
    return load().moe_block_workspace_size(T, H, I, E, K)


def moe_forward_block(x, logits, bias, w13, s13, w2, s2, n_shared, num_groups, topk_group, top_k,
                      scoring=SIGMOID, renormalize=True, routed_scaling_factor=1.0, out=None,
                      workspace=None, stream=None):
    """The layer in block FP8: s13 [E+n_shared, 2I/128, H/128], s2 [E+n_shared, H/128, I/128]."""
    import torch
    _need_cuda(x, logits, bias, w13, s13, w2, s2, out, workspace)
    T, H, I, E = _dims(x, logits, w13, w2, n_shared)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device) if out is None else out
    _need_buf("moe_forward_block", "out", out, T * H, (torch.bfloat16,))
    if workspace is None:
        nws = moe_block_workspace_size(T, H, I, E + n_shared, top_k + n_shared)
        workspace = torch.empty(nws, dtype=torch.uint8, device=x.device)
    _check("moe_forward_block", load().moe_forward_block(
        _ptr(x), _ptr(logits), _ptr(bias), _ptr(_u8(w13)), _ptr(s13), _ptr(_u8(w2)), _ptr(s2),
        T, H, I, E, int(n_shared), num_groups, topk_group, top_k, scoring,
        int(bool(renormalize)), float(routed_scaling_factor), _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def moe_forward_block_host(x_host, logits_host, bias, w13, s13, w2, s2, n_shared, num_groups,
                           topk_group, top_k, scoring, renormalize, routed_scaling_factor,
                           out_host, workspace, stream=None):
    """moe_forward_block with x, logits and out in host memory."""
    _need_cuda(bias, w13, s13, w2, s2, workspace)
    for t in (x_host, logits_host, out_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("moe_forward_block_host: x, logits and out must be contiguous "
                             "host tensors")
    T, H, I, E = _dims(x_host, logits_host, w13, w2, n_shared)
    _check("moe_forward_block_host", load().moe_forward_block_host(
        _ptr(x_host), _ptr(logits_host), _ptr(bias), _ptr(_u8(w13)), _ptr(s13), _ptr(_u8(w2)),
        _ptr(s2), T, H, I, E, int(n_shared), num_groups, topk_group, top_k, scoring,
        int(bool(renormalize)), float(routed_scaling_factor), _ptr(out_host), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out_host


# ---- NVFP4 (E2M1 codes two per byte, E4M3 scale per 16 along K, fp32 global)
def moe_permute_quant_nvfp4(x, topk_ids, E, g, workspace=None, stream=None, a_q=None, sf=None,
                            src2dst=None, offsets=None):
    """Pre-reorder with NVFP4 quantisation (global scale g). Returns (a_q
    [T*K, H/2] packed, sf [T*K, H/16], src2dst, offsets); given buffers are
    filled in place."""
    import torch
    _need_cuda(x, topk_ids, workspace, a_q, sf, src2dst, offsets)
    T, H = x.shape
    K = topk_ids.shape[1]
    dev = x.device
    M = T * K
    a_q = torch.empty((M, H // 2), dtype=torch.uint8, device=dev) if a_q is None else a_q
    sf = torch.empty((M, H // 16), dtype=torch.uint8, device=dev) if sf is None else sf
    src2dst = torch.empty(M, dtype=torch.int32, device=dev) if src2dst is None else src2dst
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    fn = "moe_permute_quant_nvfp4"
    _need_buf(fn, "a_q", a_q, M * (H // 2), (torch.uint8,))
    _need_buf(fn, "sf", sf, M * (H // 16), (torch.uint8,))
    _need_buf(fn, "src2dst", src2dst, M, (torch.int32,))
    _need_buf(fn, "offsets", offsets, E + 1, (torch.int32,))
    if workspace is None:
        workspace = torch.empty(max(moe_permute_workspace_size(T, E, K), 256), dtype=torch.uint8,
                                device=dev)
    _check("moe_permute_quant_nvfp4", load().moe_permute_quant_nvfp4(
        _ptr(x), _ptr(topk_ids), T, H, E, K, float(g), _ptr(a_q), _ptr(sf), _ptr(src2dst),
        _ptr(offsets), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return a_q, sf, src2dst, offsets


def moe_act_quant_nvfp4(h, g, stream=None, q=None, sf=None):
    """NVFP4 requantisation of h [M, I] bf16: (q [M, I/2] packed, sf [M, I/16]);
    given buffers are filled in place."""
    import torch
    _need_cuda(h, q, sf)
    M, I = h.shape
    q = torch.empty((M, I // 2), dtype=torch.uint8, device=h.device) if q is None else q
    sf = torch.empty((M, I // 16), dtype=torch.uint8, device=h.device) if sf is None else sf
    _need_buf("moe_act_quant_nvfp4", "q", q, M * (I // 2), (torch.uint8,))
    _need_buf("moe_act_quant_nvfp4", "sf", sf, M * (I // 16), (torch.uint8,))
    _check("moe_act_quant_nvfp4", load().moe_act_quant_nvfp4(
        _ptr(h), M, I, float(g), _ptr(q), _ptr(sf), _stream(stream)))
    return q, sf


def moe_nvfp4_arrange_scales(sb, epilogue, stream=None):
    """Weight block scales [E, N, Kd/16] -> the GEMM's copy order (same shape)."""
    import torch
    _need_cuda(sb)
    E, N, ks = sb.shape
    out = torch.empty_like(sb)
    _check("moe_nvfp4_arrange_scales", load().moe_nvfp4_arrange_scales(
        _ptr(sb), E, N, ks * 16, epilogue, _ptr(out), _stream(stream)))
    return out


def moe_grouped_gemm_nvfp4(A, sfa, ga, B, sfb, gb, offsets, epilogue=EPI_BF16, C=None,
                           stream=None):
    """A [M, Kd/2] packed, sfa [M, Kd/16]; B [E, N, Kd/2] packed, sfb [E, N, Kd/16]
    arranged by moe_nvfp4_arrange_scales (same epilogue), gb [E]; ga a float."""
    import torch
    _need_cuda(A, sfa, B, sfb, gb, offsets, C)
    M = A.shape[0]
    E, N, kb = B.shape
    Kd = 2 * kb
    cols = N // 2 if epilogue == EPI_SILU_MUL else N
    if C is None:
        C = torch.empty((M, cols), dtype=torch.bfloat16, device=A.device)
    _gemm_bufs("moe_grouped_gemm_nvfp4", M, N, E, cols, sfa, M * (Kd // 16), sfb,
               E * N * (Kd // 16), offsets, C, None, scale_dtypes=(torch.uint8,))
    _need_buf("moe_grouped_gemm_nvfp4", "gb", gb, E, (torch.float32,))
    _check("moe_grouped_gemm_nvfp4", load().moe_grouped_gemm_nvfp4(
        _ptr(A), _ptr(sfa), float(ga), _ptr(B), _ptr(sfb), _ptr(gb), _ptr(offsets), M, N, Kd, E,
        epilogue, _ptr(C), _stream(stream)))
    return C


def moe_nvfp4_workspace_size(T, H, I, E, K):
    return load().moe_nvfp4_workspace_size(T, H, I, E, K)


def moe_forward_nvfp4(x, logits, bias, w13, s13, g13, w2, s2, g2, ga1, ga2, n_shared,
                      num_groups, topk_group, top_k, scoring=SIGMOID, renormalize=True,
                      routed_scaling_factor=1.0, out=None, workspace=None, stream=None):
    """The layer in NVFP4: w13 [E+S, 2I, H/2], s13 [E+S, 2I, H/16], g13 [E+S];
    w2 [E+S, H, I/2], s2 [E+S, H, I/16], g2 [E+S]; ga1, ga2 floats."""
    import torch
    _need_cuda(x, logits, bias, w13, s13, g13, w2, s2, g2, out, workspace)
    T, H = x.shape
    E = logits.shape[1]
    I = w2.shape[2] * 2
    out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device) if out is None else out
    _need_buf("moe_forward_nvfp4", "out", out, T * H, (torch.bfloat16,))
    if workspace is None:
        nws = moe_nvfp4_workspace_size(T, H, I, E + n_shared, top_k + n_shared)
        workspace = torch.empty(nws, dtype=torch.uint8, device=x.device)
    _check("moe_forward_nvfp4", load().moe_forward_nvfp4(
        _ptr(x), _ptr(logits), _ptr(bias), _ptr(w13), _ptr(s13), _ptr(g13), _ptr(w2), _ptr(s2),
        _ptr(g2), float(ga1), float(ga2), T, H, I, E, int(n_shared), num_groups, topk_group,
        top_k, scoring, int(bool(renormalize)), float(routed_scaling_factor), _ptr(out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def moe_forward_nvfp4_host(x_host, logits_host, bias, w13, s13, g13, w2, s2, g2, ga1, ga2,
                           n_shared, num_groups, topk_group, top_k, scoring, renormalize,
                           routed_scaling_factor, out_host, workspace, stream=None):
    """moe_forward_nvfp4 with x, logits and out in host memory."""
    _need_cuda(bias, w13, s13, g13, w2, s2, g2, workspace)
    for t in (x_host, logits_host, out_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("moe_forward_nvfp4_host: x, logits and out must be contiguous "
                             "host tensors")
    T, H = x_host.shape
    E = logits_host.shape[1]
    I = w2.shape[2] * 2
    _check("moe_forward_nvfp4_host", load().moe_forward_nvfp4_host(
        _ptr(x_host), _ptr(logits_host), _ptr(bias), _ptr(w13), _ptr(s13), _ptr(g13), _ptr(w2),
        _ptr(s2), _ptr(g2), float(ga1), float(ga2), T, H, I, E, int(n_shared), num_groups,
        topk_group, top_k, scoring, int(bool(renormalize)), float(routed_scaling_factor),
        _ptr(out_host), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out_host


def moe_test_gemm_timeout(A, scale_a, B, scale_b, offsets, epilogue, C, stall_stage,
                          stream=None):
    """Failure-detection test: one pipeline stage of CTA 0 never receives its
    bytes, so the GEMM's bounded waits run out (~2 s); moe_device_status()
    then returns DEV_PIPE_TIMEOUT and the context stays usable."""
    _need_cuda(A, scale_a, B, scale_b, offsets, C)
    M, Kd = A.shape
    E, N, _ = B.shape
    _check("moe_test_gemm_timeout", load().moe_test_gemm_timeout(
        _ptr(_u8(A)), _ptr(scale_a), _ptr(_u8(B)), _ptr(scale_b), _ptr(offsets), M, N, Kd, E,
        epilogue, _ptr(C), int(stall_stage), _stream(stream)))
    return C


def moe_test_gemm_nvfp4_timeout(A, sfa, ga, B, sfb, gb, offsets, epilogue, C, stall_stage,
                                stream=None):
    """moe_test_gemm_timeout for the NVFP4 GEMM (A [M, Kd/2] and B [E, N, Kd/2]
    packed, sfb arranged): one pipeline stage of CTA 0 never receives its
    bytes, the waits run out (~2 s), moe_device_status() then returns
    DEV_PIPE_TIMEOUT and the context stays usable."""
    _need_cuda(A, sfa, B, sfb, gb, offsets, C)
    M, Kd = A.shape[0], A.shape[1] * 2
    E, N = B.shape[0], B.shape[1]
    _check("moe_test_gemm_nvfp4_timeout", load().moe_test_gemm_nvfp4_timeout(
        _ptr(A), _ptr(sfa), float(ga), _ptr(B), _ptr(sfb), _ptr(gb), _ptr(offsets), M, N, Kd, E,
        epilogue, _ptr(C), int(stall_stage), _stream(stream)))
    return C


def moe_device_status():
    """Synchronise the device and return (and clear) its device error code."""
    code = ctypes.c_int(0)
    st = load().moe_device_status(ctypes.byref(code))
    if st not in (0, -5):
        raise MoEError("moe_device_status", st)
    return code.value


def moe_pipeline_workspace_size(desc):
    return load().moe_pipeline_workspace_size(ctypes.byref(desc))


def moe_forward_host_pipelined(desc, x_hosts, logits_hosts, out_hosts, workspace, stream=None):
    """n batches of host tensors (x [T,H] bf16, logits [T,E] f32 in, out
    [T,H] bf16 out; pinned for the copies to overlap the compute) through the
    layer `desc`, with batch i+1's inputs and batch i-1's output crossing the
    host link while batch i computes."""
    n = len(x_hosts)
    if not (len(logits_hosts) == n == len(out_hosts)) or n < 1:
        raise ValueError("moe_forward_host_pipelined: one x, logits and out per batch")
    for t in list(x_hosts) + list(logits_hosts) + list(out_hosts):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("moe_forward_host_pipelined: host tensors, contiguous")
    arr = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])  # noqa: E731
    xs, ls, os_ = arr(x_hosts), arr(logits_hosts), arr(out_hosts)
    _check("moe_forward_host_pipelined", load().moe_forward_host_pipelined(
        ctypes.byref(desc), n, ctypes.cast(xs, _P), ctypes.cast(ls, _P), ctypes.cast(os_, _P),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out_hosts


class MoELayer:
    """A layer's resident weights plus a reusable workspace; calls moe_forward
    (moe_forward_shared when the layer has shared experts, stored as the last
    n_shared experts of w13/w2; moe_forward_block for block-quantised weights,
    quant="block")."""

    def __init__(self, w13, s13, w2, s2, bias, num_groups, topk_group, top_k, scoring,
                 renormalize, routed_scaling_factor, max_tokens, n_shared=0, quant="token",
                 nvfp4=None):
        """quant="nvfp4": w13/w2 hold packed E2M1 codes and s13/s2 E4M3 block
        scales; nvfp4 = dict(g13=..., g2=..., ga1=..., ga2=...) the global
        scales."""
        import torch
        if quant not in ("token", "block", "nvfp4"):
            raise ValueError("MoELayer: quant is 'token', 'block' or 'nvfp4'")
        self.quant = quant
        self.w13, self.s13, self.w2, self.s2, self.bias = w13, s13, w2, s2, bias
        EA, I2, self.H = w13.shape
        if quant == "nvfp4":
            self.H *= 2  # two codes per byte
            self.g13, self.g2 = nvfp4["g13"], nvfp4["g2"]
            self.ga1, self.ga2 = float(nvfp4["ga1"]), float(nvfp4["ga2"])
            # the weights' block scales in the order the GEMMs copy them (the
            # row-major ones stay in s13_rows / s2_rows)
            self.s13_rows, self.s2_rows = s13, s2
            self.s13 = moe_nvfp4_arrange_scales(s13, EPI_SILU_MUL)
            self.s2 = moe_nvfp4_arrange_scales(s2, EPI_BF16)
        self.n_shared = n_shared
        self.E = EA - n_shared  # routed experts
        self.I = I2 // 2
        self.num_groups, self.topk_group, self.top_k = num_groups, topk_group, top_k
        self.scoring, self.renormalize, self.rsf = scoring, renormalize, routed_scaling_factor
        self.max_tokens = max_tokens
        size = {"block": moe_block_workspace_size, "nvfp4": moe_nvfp4_workspace_size}.get(
            quant, moe_workspace_size)
        self.workspace = torch.empty(size(max_tokens, self.H, self.I, EA, top_k + n_shared),
                                     dtype=torch.uint8, device=w13.device)

    def __call__(self, x, logits, out=None, stream=None):
        if x.shape[0] > self.max_tokens:
            raise ValueError("MoELayer: more tokens than the workspace was sized for")
        if self.quant == "nvfp4":
            return moe_forward_nvfp4(x, logits, self.bias, self.w13, self.s13, self.g13, self.w2,
                                     self.s2, self.g2, self.ga1, self.ga2, self.n_shared,
                                     self.num_groups, self.topk_group, self.top_k, self.scoring,
                                     self.renormalize, self.rsf, out=out,
                                     workspace=self.workspace, stream=stream)
        if self.quant == "block":
            return moe_forward_block(x, logits, self.bias, self.w13, self.s13, self.w2, self.s2,
                                     self.n_shared, self.num_groups, self.topk_group,
                                     self.top_k, self.scoring, self.renormalize, self.rsf,
                                     out=out, workspace=self.workspace, stream=stream)
        if self.n_shared:
            return moe_forward_shared(x, logits, self.bias, self.w13, self.s13, self.w2,
                                      self.s2, self.n_shared, self.num_groups, self.topk_group,
                                      self.top_k, self.scoring, self.renormalize, self.rsf,
                                      out=out, workspace=self.workspace, stream=stream)
        return moe_forward(x, logits, self.bias, self.w13, self.s13, self.w2, self.s2,
                           self.num_groups, self.topk_group, self.top_k, self.scoring,
                           self.renormalize, self.rsf, out=out, workspace=self.workspace,
                           stream=stream)

    def capture(self, x, logits, out):
        """Records one forward on the fixed device buffers x, logits and out
        into a CUDA graph and returns it (torch.cuda.CUDAGraph); g.replay()
        reruns the layer on whatever those buffers hold, launching the same
        kernels without per-call host work. One eager call first, outside the
        capture, does the per-device set-up (kernel attributes, TMA
        descriptors, the device error word)."""
        import torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self(x, logits, out=out)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self(x, logits, out=out)
        return g

    def desc(self, T):
        """The struct moe_layer of this layer for batches of T tokens."""
        q = {"token": QUANT_TOKEN, "block": QUANT_BLOCK, "nvfp4": QUANT_NVFP4}[self.quant]
        fp4 = self.quant == "nvfp4"
        v = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        return MoELayerDesc(q, T, self.H, self.I, self.E, self.n_shared, self.num_groups,
                            self.topk_group, self.top_k, self.scoring, int(self.renormalize),
                            self.rsf, v(self.bias), v(self.w13), v(self.s13), v(self.w2),
                            v(self.s2), v(self.g13) if fp4 else None,
                            v(self.g2) if fp4 else None, self.ga1 if fp4 else 0.0,
                            self.ga2 if fp4 else 0.0)

    def forward_host_pipelined(self, x_hosts, logits_hosts, out_hosts, stream=None):
        """Batches from host memory through moe_forward_host_pipelined (copies
        overlapped with the compute); the pipeline workspace is kept per T."""
        import torch
        T = x_hosts[0].shape[0]
        d = self.desc(T)
        ws = getattr(self, "_pipe_ws", None)
        need = moe_pipeline_workspace_size(d)
        if need == 0:
            raise MoEError("moe_pipeline_workspace_size", -1)
        if ws is None or ws.numel() < need:
            ws = self._pipe_ws = torch.empty(need, dtype=torch.uint8, device=self.w13.device)
        return moe_forward_host_pipelined(d, x_hosts, logits_hosts, out_hosts, ws, stream)

    def forward_host(self, x_host, logits_host, out_host, stream=None):
        if self.quant == "nvfp4":
            return moe_forward_nvfp4_host(x_host, logits_host, self.bias, self.w13, self.s13,
                                          self.g13, self.w2, self.s2, self.g2, self.ga1,
                                          self.ga2, self.n_shared, self.num_groups,
                                          self.topk_group, self.top_k, self.scoring,
                                          self.renormalize, self.rsf, out_host,
                                          self.workspace, stream=stream)
        if self.quant == "block":
            return moe_forward_block_host(x_host, logits_host, self.bias, self.w13, self.s13,
                                          self.w2, self.s2, self.n_shared, self.num_groups,
                                          self.topk_group, self.top_k, self.scoring,
                                          self.renormalize, self.rsf, out_host,
                                          self.workspace, stream=stream)
        if self.n_shared:
            return moe_forward_shared_host(x_host, logits_host, self.bias, self.w13, self.s13,
                                           self.w2, self.s2, self.n_shared, self.num_groups,
                                           self.topk_group, self.top_k, self.scoring,
                                           self.renormalize, self.rsf, out_host,
                                           self.workspace, stream=stream)
        return moe_forward_host(x_host, logits_host, self.bias, self.w13, self.s13, self.w2,
                                self.s2, self.num_groups, self.topk_group, self.top_k,
                                self.scoring, self.renormalize, self.rsf, out_host,
                                self.workspace, stream=stream)


from .ep import (EPMoELayer, moe_ep_combine, moe_ep_dispatch, moe_ep_expert_forward,  # noqa: E402
                 moe_ep_recv_reorder, moe_ep_return_gather)
