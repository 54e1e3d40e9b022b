"""Routing structure of the synthetic workloads (CPU): the gate of the oracle
on each workload's seeded logits and bias gives the expert loads that the
input recipe promises (partial activation at decode, every expert busy at
prefill, the two skewed layers' hot shares)."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from moe_expert_layer_grouped_gb300 import synth  # noqa: E402


def _loads(name, seed=0):
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, seed, weights=False)
    bias = None if d["bias"] is None else d["bias"].numpy()
    ids, _ = oracle.gate(d["logits"].numpy(), bias, wl.num_groups, wl.topk_group, wl.top_k,
                         wl.scoring, wl.renormalize, wl.rsf)
    return wl, ids, np.bincount(ids.ravel(), minlength=wl.E)


def test_decode_activates_part_of_the_experts():
    # 128 tokens x 8 picks over 256 experts under a shared N(0, 0.1) bias:
    # a GEMM step reads only the active experts' weights
    _, _, cnt = _loads("dsv3_decode_t128")
    assert 120 <= np.count_nonzero(cnt) <= 200
    assert cnt.sum() == 128 * 8


@pytest.mark.parametrize("name,E,lo,hi", [("dsv3_prefill_t8192", 256, 150, 400),
                                           ("mixtral_t4096", 8, 800, 1300)])
def test_prefill_keeps_every_expert_busy(name, E, lo, hi):
    _, _, cnt = _loads(name)
    assert cnt.shape[0] == E and lo <= cnt.min() and cnt.max() <= hi


def test_skewed_literal_bias_sends_every_token_to_the_hot_experts():
    # +3.0 on the 26 experts with e % 10 == 0 outweighs any sigmoid score, and
    # each of the 4 kept groups holds at least three of them
    _, ids, cnt = _loads("dsv3_skewed_t16384")
    assert np.all(ids % 10 == 0)
    assert np.count_nonzero(cnt) == 26


def test_skewed_half_bias_splits_about_half_to_the_hot_experts():
    wl, ids, cnt = _loads("dsv3_skewed_half_t16384")
    assert wl.hot_bias == pytest.approx(0.225)
    share = np.mean(ids % 10 == 0)
    assert 0.45 <= share <= 0.55, share
    assert not np.any(ids % 8 == 7)          # the -10 experts are never taken
    assert 150 <= np.count_nonzero(cnt) < 230
    hot = cnt[np.arange(wl.E) % 10 == 0]
    assert hot.min() > 4 * np.median(cnt[cnt > 0])  # hot experts several times the typical load
