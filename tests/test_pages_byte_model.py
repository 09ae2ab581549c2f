"""The expert blob byte model against the sizes printed on the pages (tests/golden)."""
import json
import os

from routed_expert_ffn_grouped_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_byte_model.json")


def _load():
    with open(GOLDEN) as f:
        return json.load(f)


def _close(got, entry):
    return abs(got - entry["value"]) <= entry["rel_tol"] * entry["value"]


def test_expert_size_matches_pages():
    g = _load()
    L = synth.blob_layout(synth.GLM52.d, synth.GLM52.ffn)
    assert L.nibble_bytes == 18_874_368
    assert _close(L.nibble_bytes, g["expert_nibble_bytes_approx"])
    e = g["all_routed_experts_bytes"]
    assert _close(e["n_experts"] * L.nibble_bytes, e)
    c = g["cold_token_read_bytes"]
    assert _close(c["n_layers"] * c["experts_per_layer"] * L.nibble_bytes, c)


def test_blob_layout_parts():
    # Full blob = nibbles + fp32 scales (one per 32 weights, 1/4 of the nibble bytes).
    for spec, total in ((synth.TINY, 245_760), (synth.OLMOE, 3_932_160), (synth.GLM52, 23_592_960)):
        L = synth.blob_layout(spec.d, spec.ffn)
        assert L.nbytes == total
        assert L.nbytes == L.nibble_bytes + L.nibble_bytes // 4
        assert L.w3 - L.w1 == L.w2 - L.w3 == spec.d * spec.ffn // 2
        assert all(o % 256 == 0 for o in (L.w1, L.w3, L.w2, L.s1, L.s3, L.s2))
