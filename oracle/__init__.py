"""numpy front end of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` import this module. The product library never
does.

Every function takes and returns numpy arrays; bf16 tensors travel as their
uint16 bit patterns and FP8 e4m3 tensors as uint8 codes.
"""
import ctypes
import os

import numpy as np

from . import build as _build

SIGMOID = 0
SOFTMAX = 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        sig = {
            "oracle_set_threads": (None, [i32]),
            "oracle_get_threads": (i32, []),
            "oracle_exp32": (f32, [f32]),
            "oracle_exp32_n": (None, [P, P, i64]),
            "oracle_sigmoid32": (f32, [f32]),
            "oracle_sigmoid32_n": (None, [P, P, i64]),
            "oracle_e4m3_encode": (ctypes.c_uint8, [f32]),
            "oracle_e4m3_encode_n": (None, [P, P, i64]),
            "oracle_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_bf16_round_n": (None, [P, P, i64]),
            "oracle_gate": (i32, [P, P, i32, i32, i32, i32, i32, i32, i32, f32, P, P]),
            "oracle_route": (None, [P, i32, i32, i32, P, P]),
            "oracle_row_quant": (None, [P, i64, i32, P, P]),
            "oracle_permute_quant": (None, [P, P, i32, i32, i32, i32, P, P, P, P]),
            "oracle_grouped_gemm": (None, [P, P, P, P, P, i32, i32, i32, i32, P]),
            "oracle_silu_mul": (None, [P, i64, i32, P]),
            "oracle_unpermute_sum": (None, [P, P, P, i32, i32, i32, P]),
            "oracle_forward_tokens": (i32, [P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                            i32, i32, i32, i32, f32, P, i32, P, P, P]),
            "oracle_forward_tokens_shared": (i32, [P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                   i32, i32, i32, i32, i32, i32, f32, P, i32,
                                                   P, P, P]),
            "oracle_block_quant": (None, [P, i64, i32, P, P]),
            "oracle_permute_quant_block": (None, [P, P, i32, i32, i32, i32, P, P, P, P]),
            "oracle_grouped_gemm_block": (None, [P, P, P, P, P, i32, i32, i32, i32, P]),
            "oracle_forward_tokens_block": (i32, [P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                  i32, i32, i32, i32, i32, i32, f32, P, i32,
                                                  P, P, P]),
            "oracle_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e2m1_encode_n": (None, [P, P, i64]),
            "oracle_nvfp4_quant": (None, [P, i64, i32, f32, P, P]),
            "oracle_grouped_gemm_nvfp4": (None, [P, P, f32, P, P, P, P, i32, i32, i32, i32, P]),
            "oracle_forward_tokens_nvfp4": (i32, [P, P, P, P, P, P, P, P, P, f32, f32, i32, i32,
                                                  i32, i32, i32, i32, i32, i32, i32, i32, f32,
                                                  P, i32, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n):
    lib().oracle_set_threads(int(n))


def get_threads():
    return lib().oracle_get_threads()


def exp32(x):
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib().oracle_exp32_n(_p(x), _p(y), x.size)
    return y


def sigmoid32(x):
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib().oracle_sigmoid32_n(_p(x), _p(y), x.size)
    return y


def e4m3_encode(x):
    x = _c(x, np.float32)
    q = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_encode_n(_p(x), _p(q), x.size)
    return q


def e4m3_decode_table():
    L = lib()
    return np.array([L.oracle_e4m3_decode(i) for i in range(256)], np.float64)


def e4m3_decode(q):
    return e4m3_decode_table()[np.asarray(q, np.uint8)]


def bf16_round(v):
    """fp64 values -> bf16 bit patterns (uint16), round to nearest even."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_bf16_round_n(_p(v), _p(out), v.size)
    return out


def bf16_to_f64(bits):
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def gate(logits, bias, num_groups, topk_group, top_k, scoring=SIGMOID,
         renormalize=True, routed_scaling_factor=1.0):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float32)
    rc = lib().oracle_gate(_p(logits), _p(b), T, E, num_groups, topk_group, top_k,
                           scoring, int(bool(renormalize)), float(routed_scaling_factor),
                           _p(ids), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_gate: status {rc}")
    return ids, w


def route(topk_ids, E):
    ids = _c(topk_ids, np.int32)
    T, K = ids.shape
    offsets = np.empty(E + 1, np.int32)
    src2dst = np.empty(T * K, np.int32)
    lib().oracle_route(_p(ids), T, E, K, _p(offsets), _p(src2dst))
    return offsets, src2dst


def row_quant(x_bits):
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty(R, np.float32)
    lib().oracle_row_quant(_p(x), R, C, _p(q), _p(s))
    return q, s


def permute_quant(x_bits, topk_ids, E):
    x = _c(x_bits, np.uint16)
    ids = _c(topk_ids, np.int32)
    T, H = x.shape
    K = ids.shape[1]
    M = T * K
    a_q = np.empty((M, H), np.uint8)
    sa = np.empty(M, np.float32)
    src2dst = np.empty(M, np.int32)
    offsets = np.empty(E + 1, np.int32)
    lib().oracle_permute_quant(_p(x), _p(ids), T, H, E, K, _p(a_q), _p(sa), _p(src2dst),
                               _p(offsets))
    return a_q, sa, src2dst, offsets


def grouped_gemm(A, scale_a, B, scale_b, offsets):
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(scale_a, np.float32)
    sb = _c(scale_b, np.float32)
    off = _c(offsets, np.int32)
    M, Kd = A.shape
    E, N, Kd2 = B.shape
    assert Kd == Kd2 and off.size == E + 1
    C = np.empty((M, N), np.float64)
    lib().oracle_grouped_gemm(_p(A), _p(sa), _p(B), _p(sb), _p(off), M, N, Kd, E, _p(C))
    return C


def silu_mul(C):
    C = _c(C, np.float64)
    M, N2 = C.shape
    I = N2 // 2
    h = np.empty((M, I), np.float64)
    lib().oracle_silu_mul(_p(C), M, I, _p(h))
    return h


def act_quant(h_bits):
    """Per-row requantisation of bf16 h (bit patterns) -> (codes, scales)."""
    return row_quant(h_bits)


def unpermute_sum(down, src2dst, topk_w):
    down = _c(down, np.float64)
    s2d = _c(src2dst, np.int32)
    w = _c(topk_w, np.float32)
    T, K = w.shape
    H = down.shape[1]
    out = np.empty((T, H), np.float64)
    lib().oracle_unpermute_sum(_p(down), _p(s2d), _p(w), T, K, H, _p(out))
    return out


def forward_tokens(x_bits, logits, bias, w13, s13, w2, s2, num_groups, topk_group,
                   top_k, scoring, renormalize, routed_scaling_factor, tokens=None,
                   n_shared=0):
    """Whole layer for the listed tokens (all tokens when None).

    With n_shared > 0, w13/w2 (and their scales) hold E + n_shared experts, the
    last n_shared being shared experts that every token adds with weight 1.
    Returns (out [n,H] fp64, ids [n,K], w [n,K]) (routed slots only)."""
    x = _c(x_bits, np.uint16)
    logits = _c(logits, np.float32)
    T, H = x.shape
    E = logits.shape[1]
    I = w2.shape[2]
    assert w13.shape == (E + n_shared, 2 * I, H) and w2.shape == (E + n_shared, H, I)
    b = None if bias is None else _c(bias, np.float32)
    tok = np.arange(T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    n = tok.size
    out = np.empty((n, H), np.float64)
    ids = np.empty((n, top_k), np.int32)
    w = np.empty((n, top_k), np.float32)
    w13 = _c(w13, np.uint8)
    w2 = _c(w2, np.uint8)
    s13 = _c(s13, np.float32)
    s2 = _c(s2, np.float32)
    rc = lib().oracle_forward_tokens_shared(_p(x), _p(logits), _p(b), _p(w13), _p(s13),
                                            _p(w2), _p(s2), T, H, I, E, int(n_shared),
                                            num_groups, topk_group, top_k, scoring,
                                            int(bool(renormalize)),
                                            float(routed_scaling_factor), _p(tok), n, _p(out),
                                            _p(ids), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_forward_tokens: status {rc}")
    return out, ids, w


def forward_steps(x_bits, logits, bias, w13, s13, w2, s2, num_groups, topk_group, top_k,
                  scoring, renormalize, routed_scaling_factor, n_shared=0):
    """The layer step by step over all tokens, returning every intermediate
    (small configurations only: materialises [M, 2I] in fp64). Shared experts
    (n_shared > 0) take slots K .. K+n_shared-1 of every token, ids E.., weight 1."""
    E = logits.shape[1]
    ids, w = gate(logits, bias, num_groups, topk_group, top_k, scoring, renormalize,
                  routed_scaling_factor)
    if n_shared:
        T = ids.shape[0]
        ids = np.concatenate([ids, np.broadcast_to(
            np.arange(E, E + n_shared, dtype=np.int32), (T, n_shared))], axis=1)
        w = np.concatenate([w, np.ones((T, n_shared), np.float32)], axis=1)
        E += n_shared
    a_q, sa, src2dst, offsets = permute_quant(x_bits, ids, E)
    C13 = grouped_gemm(a_q, sa, w13, s13, offsets)
    h = silu_mul(C13)
    h_bits = bf16_round(h)
    q2, sa2 = act_quant(h_bits)
    down = grouped_gemm(q2, sa2, w2, s2, offsets)
    out = unpermute_sum(down, src2dst, w)
    return dict(ids=ids, w=w, a_q=a_q, scale_a=sa, src2dst=src2dst, offsets=offsets,
                c13=C13, h=h, h_bits=h_bits, q2=q2, scale_a2=sa2, down=down, out=out)


# ---------------------------------------------------------------------------
# block-quantised FP8: 128-channel activation blocks, 128 x 128 weight blocks
# ---------------------------------------------------------------------------
QB = 128


def block_quant(x_bits):
    """bf16 [R,C] (bit patterns) -> (e4m3 codes [R,C], scales [R, C/128])."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert C % QB == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // QB), np.float32)
    lib().oracle_block_quant(_p(x), R, C, _p(q), _p(s))
    return q, s


def permute_quant_block(x_bits, topk_ids, E):
    x = _c(x_bits, np.uint16)
    ids = _c(topk_ids, np.int32)
    T, H = x.shape
    K = ids.shape[1]
    M = T * K
    a_q = np.empty((M, H), np.uint8)
    sa = np.empty((M, H // QB), np.float32)
    src2dst = np.empty(M, np.int32)
    offsets = np.empty(E + 1, np.int32)
    lib().oracle_permute_quant_block(_p(x), _p(ids), T, H, E, K, _p(a_q), _p(sa), _p(src2dst),
                                     _p(offsets))
    return a_q, sa, src2dst, offsets


def grouped_gemm_block(A, scale_a, B, scale_b, offsets):
    """scale_a [M, Kd/128]; scale_b [E, N/128, Kd/128]; fp64 result [M, N]."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(scale_a, np.float32)
    sb = _c(scale_b, np.float32)
    off = _c(offsets, np.int32)
    M, Kd = A.shape
    E, N, Kd2 = B.shape
    assert Kd == Kd2 and off.size == E + 1 and Kd % QB == 0 and N % QB == 0
    assert sa.shape == (M, Kd // QB) and sb.shape == (E, N // QB, Kd // QB)
    C = np.empty((M, N), np.float64)
    lib().oracle_grouped_gemm_block(_p(A), _p(sa), _p(B), _p(sb), _p(off), M, N, Kd, E, _p(C))
    return C


def forward_tokens_block(x_bits, logits, bias, w13, s13, w2, s2, num_groups, topk_group, top_k,
                         scoring, renormalize, routed_scaling_factor, tokens=None, n_shared=0):
    """Whole layer in block FP8 for the listed tokens: s13 [E+S, 2I/128, H/128],
    s2 [E+S, H/128, I/128]. Returns (out [n,H] fp64, ids [n,K], w [n,K])."""
    x = _c(x_bits, np.uint16)
    logits = _c(logits, np.float32)
    T, H = x.shape
    E = logits.shape[1]
    I = w2.shape[2]
    n = E + n_shared
    assert w13.shape == (n, 2 * I, H) and w2.shape == (n, H, I)
    assert s13.shape == (n, 2 * I // QB, H // QB) and s2.shape == (n, H // QB, I // QB)
    b = None if bias is None else _c(bias, np.float32)
    tok = np.arange(T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    nt = tok.size
    out = np.empty((nt, H), np.float64)
    ids = np.empty((nt, top_k), np.int32)
    w = np.empty((nt, top_k), np.float32)
    w13, w2 = _c(w13, np.uint8), _c(w2, np.uint8)
    s13, s2 = _c(s13, np.float32), _c(s2, np.float32)
    rc = lib().oracle_forward_tokens_block(_p(x), _p(logits), _p(b), _p(w13), _p(s13), _p(w2),
                                           _p(s2), T, H, I, E, int(n_shared), num_groups,
                                           topk_group, top_k, scoring, int(bool(renormalize)),
                                           float(routed_scaling_factor), _p(tok), nt, _p(out),
                                           _p(ids), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_forward_tokens_block: status {rc}")
    return out, ids, w


def forward_steps_block(x_bits, logits, bias, w13, s13, w2, s2, num_groups, topk_group, top_k,
                        scoring, renormalize, routed_scaling_factor, n_shared=0):
    """The block-FP8 layer step by step over all tokens (small configurations)."""
    E = logits.shape[1]
    ids, w = gate(logits, bias, num_groups, topk_group, top_k, scoring, renormalize,
                  routed_scaling_factor)
    if n_shared:
        T = ids.shape[0]
        ids = np.concatenate([ids, np.broadcast_to(
            np.arange(E, E + n_shared, dtype=np.int32), (T, n_shared))], axis=1)
        w = np.concatenate([w, np.ones((T, n_shared), np.float32)], axis=1)
        E += n_shared
    a_q, sa, src2dst, offsets = permute_quant_block(x_bits, ids, E)
    C13 = grouped_gemm_block(a_q, sa, w13, s13, offsets)
    h = silu_mul(C13)
    h_bits = bf16_round(h)
    q2, sa2 = block_quant(h_bits)
    down = grouped_gemm_block(q2, sa2, w2, s2, offsets)
    out = unpermute_sum(down, src2dst, w)
    return dict(ids=ids, w=w, a_q=a_q, scale_a=sa, src2dst=src2dst, offsets=offsets,
                c13=C13, h=h, h_bits=h_bits, q2=q2, scale_a2=sa2, down=down, out=out)


# ---------------------------------------------------------------------------
# NVFP4: E2M1 codes (one per byte, 0..15), one E4M3 block scale per 16
# elements along K, one fp32 global scale per tensor
# ---------------------------------------------------------------------------
FB = 16


def e2m1_decode_table():
    """Value of each of the 16 E2M1 codes (fp64)."""
    return np.array([lib().oracle_e2m1_decode(q) for q in range(16)], np.float64)


def e2m1_decode(q):
    return e2m1_decode_table()[np.asarray(q, np.uint8) & 0xF]


def e2m1_encode(x):
    x = _c(x, np.float32)
    q = np.empty(x.shape, np.uint8)
    lib().oracle_e2m1_encode_n(_p(x), _p(q), x.size)
    return q


def nvfp4_quant(x_bits, g):
    """bf16 [R,C] (bit patterns), global scale g > 0 -> (E2M1 codes [R,C],
    E4M3 block-scale codes [R, C/16])."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert C % FB == 0 and g > 0
    q = np.empty((R, C), np.uint8)
    sb = np.empty((R, C // FB), np.uint8)
    lib().oracle_nvfp4_quant(_p(x), R, C, float(g), _p(q), _p(sb))
    return q, sb


def grouped_gemm_nvfp4(A, sa, ga, B, sb, gb, offsets):
    """A [M,Kd] and B [E,N,Kd] E2M1 codes; sa [M,Kd/16] and sb [E,N,Kd/16]
    E4M3 codes; ga the activations' global scale, gb [E] the weights'.
    Returns the fp64 product [M, N]."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sa = _c(sa, np.uint8)
    sb = _c(sb, np.uint8)
    gb = _c(gb, np.float32)
    off = _c(offsets, np.int32)
    M, Kd = A.shape
    E, N, Kd2 = B.shape
    assert Kd == Kd2 and off.size == E + 1 and Kd % FB == 0 and gb.shape == (E,)
    assert sa.shape == (M, Kd // FB) and sb.shape == (E, N, Kd // FB)
    C = np.empty((M, N), np.float64)
    lib().oracle_grouped_gemm_nvfp4(_p(A), _p(sa), float(ga), _p(B), _p(sb), _p(gb), _p(off),
                                    M, N, Kd, E, _p(C))
    return C


def permute_quant_nvfp4(x_bits, topk_ids, E, g):
    """Pre-reorder with NVFP4 quantisation: each token quantised once (global
    scale g), its codes and block scales copied to the rows src2dst gives its
    K slots. Returns (codes [T*K,H], block scales [T*K,H/16], src2dst, offsets)."""
    ids = _c(topk_ids, np.int32)
    K = ids.shape[1]
    offsets, src2dst = route(ids, E)
    q, sb = nvfp4_quant(x_bits, g)
    a_q = np.empty((ids.size, q.shape[1]), np.uint8)
    sa = np.empty((ids.size, sb.shape[1]), np.uint8)
    a_q[src2dst] = np.repeat(q, K, axis=0)   # slot t*K+k holds token t
    sa[src2dst] = np.repeat(sb, K, axis=0)
    return a_q, sa, src2dst, offsets


def forward_tokens_nvfp4(x_bits, logits, bias, w13, s13, g13, w2, s2, g2, ga1, ga2, num_groups,
                         topk_group, top_k, scoring, renormalize, routed_scaling_factor,
                         tokens=None, n_shared=0):
    """Whole layer in NVFP4 for the listed tokens: codes w13 [E+S,2I,H] and
    w2 [E+S,H,I], block scales s13 [E+S,2I,H/16] and s2 [E+S,H,I/16] (E4M3
    codes), weight global scales g13, g2 [E+S], activation global scales ga1
    (x) and ga2 (h). Returns (out [n,H] fp64, ids [n,K], w [n,K])."""
    x = _c(x_bits, np.uint16)
    logits = _c(logits, np.float32)
    T, H = x.shape
    E = logits.shape[1]
    I = w2.shape[2]
    n = E + n_shared
    assert w13.shape == (n, 2 * I, H) and w2.shape == (n, H, I)
    assert s13.shape == (n, 2 * I, H // FB) and s2.shape == (n, H, I // FB)
    assert g13.shape == (n,) and g2.shape == (n,)
    b = None if bias is None else _c(bias, np.float32)
    tok = np.arange(T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    nt = tok.size
    out = np.empty((nt, H), np.float64)
    ids = np.empty((nt, top_k), np.int32)
    w = np.empty((nt, top_k), np.float32)
    w13, w2, s13, s2 = (_c(a, np.uint8) for a in (w13, w2, s13, s2))
    g13, g2 = _c(g13, np.float32), _c(g2, np.float32)
    rc = lib().oracle_forward_tokens_nvfp4(
        _p(x), _p(logits), _p(b), _p(w13), _p(s13), _p(g13), _p(w2), _p(s2), _p(g2),
        float(ga1), float(ga2), T, H, I, E, int(n_shared), num_groups, topk_group, top_k,
        scoring, int(bool(renormalize)), float(routed_scaling_factor), _p(tok), nt, _p(out),
        _p(ids), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_forward_tokens_nvfp4: status {rc}")
    return out, ids, w


def forward_steps_nvfp4(x_bits, logits, bias, w13, s13, g13, w2, s2, g2, ga1, ga2, num_groups,
                        topk_group, top_k, scoring, renormalize, routed_scaling_factor,
                        n_shared=0):
    """The NVFP4 layer step by step over all tokens (small configurations)."""
    E = logits.shape[1]
    ids, w = gate(logits, bias, num_groups, topk_group, top_k, scoring, renormalize,
                  routed_scaling_factor)
    if n_shared:
        T = ids.shape[0]
        ids = np.concatenate([ids, np.broadcast_to(
            np.arange(E, E + n_shared, dtype=np.int32), (T, n_shared))], axis=1)
        w = np.concatenate([w, np.ones((T, n_shared), np.float32)], axis=1)
        E += n_shared
    a_q, sa, src2dst, offsets = permute_quant_nvfp4(x_bits, ids, E, ga1)
    C13 = grouped_gemm_nvfp4(a_q, sa, ga1, w13, s13, g13, offsets)
    h = silu_mul(C13)
    h_bits = bf16_round(h)
    q2, sa2 = nvfp4_quant(h_bits, ga2)
    down = grouped_gemm_nvfp4(q2, sa2, ga2, w2, s2, g2, offsets)
    out = unpermute_sum(down, src2dst, w)
    return dict(ids=ids, w=w, a_q=a_q, scale_a=sa, src2dst=src2dst, offsets=offsets,
                c13=C13, h=h, h_bits=h_bits, q2=q2, scale_a2=sa2, down=down, out=out)
