"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

# Layer and GEMM outputs: max |err| <= 2e-2 * max |ref| and
# sum |err| / sum |ref| <= 5e-3 (fp32 accumulation against exact fp64).
MAX_REL = 2e-2
MEAN_REL = 5e-3


def tol_report(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    max_rel = err.max() / scale if scale > 0 else err.max()
    mean_rel = err.sum() / np.abs(ref).sum() if np.abs(ref).sum() > 0 else err.sum()
    return max_rel, mean_rel


def assert_parity(got, ref, what=""):
    max_rel, mean_rel = tol_report(got, ref)
    assert max_rel <= MAX_REL and mean_rel <= MEAN_REL, \
        f"{what}: max|err|/max|ref|={max_rel:.3e} sum|err|/sum|ref|={mean_rel:.3e}"
    return max_rel, mean_rel


def bf16_np(t):
    """bf16 torch tensor -> float64 numpy."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_bf16_to_torch(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def ragged_offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def random_e4m3(rng, shape):
    """Random FP8 codes without the NaN patterns 0x7F / 0xFF (as uint8)."""
    q = rng.integers(0, 256, shape).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] &= 0xFE
    return q


def gemm_token_tile(M, E, quant="token"):
    """Token tile of the grouped GEMM launch the library picks for M permuted
    rows over E experts: (most tokens per tile, CTA pair). Few rows per
    expert (M <= 32*E) take 64-token tiles on single CTAs in the per-token
    GEMM; otherwise it takes 256-token tiles on CTA pairs (every workload here
    has an even number of weight blocks). The block-scaled GEMM always takes
    128-token tiles (tokens are its MMA's M side) on single CTAs; the NVFP4
    GEMM 64- or 128-token tiles on single CTAs (128- or 256-row weight
    tiles: the token chunks are the same)."""
    if quant == "nvfp4":
        return (64 if M <= 32 * E else 128), False
    if quant == "block":
        return 128, False
    if M <= 32 * E:
        return 64, False
    return (256, True) if quant == "token" else (128, False)


def tile_cover_rows(offsets, bn, pair):
    """Permuted rows that put at least one compared row in every (expert,
    token chunk) tile: each chunk's first and last row and, for a CTA pair,
    the last row of the even CTA's half and the first of the odd one's.
    Chunks follow the kernel's tile table: an expert's cnt rows split into
    ceil(cnt/bn) equal chunks, rounded up to 16 rows."""
    rows = set()
    off = np.asarray(offsets, np.int64)
    for e in range(off.size - 1):
        lo_e, cnt = int(off[e]), int(off[e + 1] - off[e])
        if cnt <= 0:
            continue
        nch = -(-cnt // bn)
        csz = ((-(-cnt // nch)) + 15) // 16 * 16
        for tc in range(nch):
            lo = tc * csz
            hi = min(cnt, lo + csz)
            if lo >= hi:
                continue
            rows.update((lo_e + lo, lo_e + hi - 1))
            if pair:
                half = ((hi - lo + 31) // 32 * 32) // 2
                for r in (lo + half - 1, lo + half):
                    if lo <= r < hi:
                        rows.add(lo_e + r)
    return np.array(sorted(rows), np.int64)


def tile_cover_tokens(topk_ids, E, quant="token", n_random=40, seed=0):
    """Tokens whose outputs, compared with the oracle, exercise every tile of
    both grouped GEMMs (all weight blocks of a tile see each of its tokens):
    the tokens at tile_cover_rows, the first and last token and n_random
    more. The permutation is the oracle's (stable by expert, ascending
    token). Returns (tokens, number of tiles)."""
    import oracle
    ids = np.ascontiguousarray(topk_ids, np.int32)
    T, K = ids.shape
    offsets, src2dst = oracle.route(ids, E)
    bn, pair = gemm_token_tile(T * K, E, quant)
    rows = tile_cover_rows(offsets, bn, pair)
    row_token = np.empty(T * K, np.int64)
    row_token[src2dst] = np.arange(T * K, dtype=np.int64) // K
    rng = np.random.default_rng(seed)
    extra = rng.choice(T, min(n_random, T), replace=False)
    tokens = np.unique(np.concatenate([row_token[rows], [0, T - 1], extra]))
    cnt = np.diff(offsets.astype(np.int64))
    ntiles = int(sum(-(-c // bn) for c in cnt if c > 0))
    return tokens, ntiles
