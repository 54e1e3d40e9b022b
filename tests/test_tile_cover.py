"""The large-workload parity sample reaches every GEMM tile (CPU): the rows
it picks cover each (expert, token chunk) tile of the kernel's tile table,
its first and last row and, for CTA pairs, both CTAs' halves."""
import numpy as np

import oracle
from moe_expert_layer_grouped_gb300 import synth

from gpu_util import gemm_token_tile, tile_cover_rows, tile_cover_tokens


def _chunks(cnt, bn):
    if cnt <= 0:
        return []
    nch = -(-cnt // bn)
    csz = ((-(-cnt // nch)) + 15) // 16 * 16
    return [(tc * csz, min(cnt, (tc + 1) * csz)) for tc in range(nch) if tc * csz < cnt]


def test_every_chunk_and_half_has_a_row():
    counts = [0, 1, 15, 16, 17, 255, 256, 257, 288, 293, 511, 512, 513, 1040, 5000]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    for bn, pair in [(256, True), (128, False), (64, False)]:
        rows = set(tile_cover_rows(off, bn, pair).tolist())
        for e, cnt in enumerate(counts):
            for lo, hi in _chunks(cnt, bn):
                a, b = off[e] + lo, off[e] + hi - 1
                assert a in rows and b in rows, (bn, cnt, lo, hi)
                if pair and hi - lo > 1:
                    half = ((hi - lo + 31) // 32 * 32) // 2
                    in_even = [r for r in rows if a <= r < off[e] + lo + half]
                    in_odd = [r for r in rows if off[e] + lo + half <= r <= b]
                    assert in_even and (in_odd or lo + half >= hi), (cnt, lo, hi)
        assert all(0 <= r < off[-1] for r in rows)


def test_launch_shapes_follow_the_library():
    assert gemm_token_tile(128 * 8, 256) == (64, False)         # decode: M <= 32 E
    assert gemm_token_tile(8192 * 8, 256) == (256, True)        # prefill: CTA pairs
    assert gemm_token_tile(8192 * 8, 256, "block") == (128, False)
    assert gemm_token_tile(128 * 8, 256, "block") == (128, False)   # tokens on M at any size
    assert gemm_token_tile(128 * 8, 256, "nvfp4") == (64, False)
    assert gemm_token_tile(8192 * 8, 256, "nvfp4") == (128, False)


def test_prefill_sample_touches_every_expert_chunk():
    wl = synth.WORKLOADS["dsv3_prefill_t8192"]
    d = synth.make_inputs(wl, seed=0, device="cpu", weights=False)
    n = synth.to_numpy_inputs(d)
    ids, _ = oracle.gate(n["logits"], n["bias"], wl.num_groups, wl.topk_group, wl.top_k,
                         wl.scoring, wl.renormalize, wl.rsf)
    tokens, ntiles = tile_cover_tokens(ids, wl.E)
    off, s2d = oracle.route(ids, wl.E)
    rows_of = s2d.reshape(wl.T, wl.top_k)[tokens].ravel()
    bn, pair = gemm_token_tile(wl.T * wl.top_k, wl.E)
    for e in range(wl.E):
        for lo, hi in _chunks(int(off[e + 1] - off[e]), bn):
            seg = rows_of[(rows_of >= off[e] + lo) & (rows_of < off[e] + hi)]
            assert seg.size > 0, (e, lo, hi)
    assert ntiles >= wl.E and tokens.size < wl.T // 2
