"""The host simulation of the expert cache on the streaming workload (bench.py
--cache-sim): its operation stream follows the streaming run (one lookup batch per layer,
then the next layer's prefetch), and the library's policy on it equals the oracle's."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from routed_expert_ffn_grouped_b300 import colibri as C  # noqa: E402
from routed_expert_ffn_grouped_b300 import synth  # noqa: E402


def _ops(steps=12, predictor="previous"):
    spec = synth.GLM52
    ids, _ = synth.streaming_ids(spec, 0, bench.STREAM_LAYERS, steps + 1)
    return bench.stream_ops(ids, ids.copy(), predictor, spec.n_exp, steps), ids


def test_operation_stream_follows_the_streaming_run():
    (kinds, keys, step), ids = _ops(steps=3)
    L_, k = bench.STREAM_LAYERS, synth.GLM52.top_k
    # per layer: a batch start, k lookups, then k prefetches from the second layer call on
    assert (kinds == 0).sum() == 3 * L_ and (kinds == 1).sum() == 3 * L_ * k
    first = np.flatnonzero(kinds == 0)[1]       # start of layer 1 of step 0
    assert np.array_equal(keys[1:1 + k], ids[0, 0].astype(np.int64))   # layer 0 lookups
    assert (kinds[1 + k:first] == 2).sum() == 0  # no previous step to predict from yet
    last = np.flatnonzero(kinds == 0)[-1]        # layer 7 of step 2: prefetch layer 0 of step 3
    pre = keys[last + 1 + k:]
    assert np.array_equal(pre, ids[2, 0].astype(np.int64))


def test_policy_on_the_stream_matches_oracle(orc):
    (kinds, keys, _), _ = _ops(steps=12)
    for n_hot in (0, 64, 256):
        assert np.array_equal(C.colibri_lru_trace_hot(64, n_hot // 4, kinds, keys),
                              orc.lru_hot_trace(64, n_hot // 4, kinds, keys))
