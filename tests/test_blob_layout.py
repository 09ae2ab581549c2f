"""The stored order of expert matrices (row blocks of 32 rows, group-major inside a block),
pinned against the byte and float positions that include/colibri.h states, and round trips
between logical tensors and blobs. These are layout facts only: no arithmetic."""
import numpy as np

from routed_expert_ffn_grouped_b300 import synth


def test_nibble_positions_match_the_stated_formula():
    R, K = 96, 128                                   # 3 row blocks, 4 groups
    rng = np.random.default_rng(5)
    w = rng.integers(0, 256, (R, K // 2), dtype=np.uint8)
    flat = synth.pack_nibbles(w)
    assert flat.shape == (R * K // 2,)
    for r in (0, 1, 31, 32, 63, 95):
        for g in range(K // 32):
            base = ((r // 32) * (K // 32) + g) * 512 + (r % 32) * 16
            assert np.array_equal(flat[base:base + 16], w[r, 16 * g:16 * g + 16])


def test_scale_positions_match_the_stated_formula():
    R, K = 64, 96
    s = np.arange(R * (K // 32), dtype=np.float32).reshape(R, K // 32)
    flat = synth.pack_scales(s)
    for r in range(R):
        for g in range(K // 32):
            assert flat[((r // 32) * (K // 32) + g) * 32 + r % 32] == s[r, g]


def test_a_warp_reads_one_contiguous_group_tile():
    # group g of row block b: rows 32b..32b+31 occupy one 512-byte run, row after row
    R, K = 64, 64
    w = np.zeros((R, K // 2), np.uint8)
    for r in range(R):
        w[r, 16:32] = r                              # group 1 of every row holds its row index
    flat = synth.pack_nibbles(w)
    tile = flat[(1 * 2 + 1) * 512:(1 * 2 + 2) * 512].reshape(32, 16)
    assert np.array_equal(tile[:, 0], np.arange(32, 64))


def test_roundtrips():
    rng = np.random.default_rng(9)
    for R, K in ((32, 32), (64, 2048), (2048, 64)):
        w = rng.integers(0, 256, (R, K // 2), dtype=np.uint8)
        s = rng.standard_normal((R, K // 32)).astype(np.float32)
        assert np.array_equal(synth.unpack_nibbles(synth.pack_nibbles(w), R, K), w)
        assert np.array_equal(synth.unpack_scales(synth.pack_scales(s), R, K), s)


def test_expert_blob_roundtrip():
    spec = synth.TINY
    blob = synth.expert_blob(spec, 0, 0, 1)
    v = synth.expert_views(blob, spec.d, spec.ffn)
    assert v["w1"].shape == (spec.ffn, spec.d // 2) and v["w2"].shape == (spec.d, spec.ffn // 2)
    assert v["s2"].shape == (spec.d, spec.ffn // 32)
    again = synth.write_expert(np.empty_like(blob), spec.d, spec.ffn, v)
    assert np.array_equal(again, blob)
