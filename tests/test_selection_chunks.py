"""The chunked ranking of the decode kernel's selection (`select_cta`), restated lane by lane
on the host and checked against the textbook sequential selection: repeatedly take the best
remaining allowed expert by (score descending, index ascending).

Sigmoid routing (DeepSeek-V3 style, "Guide Complet de Colibri", router section): group
score = the sum of a group's two best biased scores, the topk_group best groups are kept,
top_k is taken inside them. Softmax routing: top_k over all experts. The kernel ranks each
group (softmax: each run of 32 experts) within itself, lists its best min(top_k, group)
experts in order, then ranks only the kept groups' listed experts against each other. The
argument that this yields the same ids is that every expert of the overall top_k is among
the best top_k of its own group under the same total order; these cases (ties, -inf scores,
one expert a group, every expert picked) check the restatement of it. GPU parity of the
kernel itself is in test_gpu_parity.py.
"""
import numpy as np
import pytest


def beats(v, i, bv, bi):
    return v > bv or (v == bv and i < bi)


def sequential(c, K, sig, NG, tg):
    """Textbook selection: the kept groups, then K times the best remaining expert."""
    E = len(c)
    if sig:
        gs = E // NG
        gsc = []
        for g in range(NG):
            vals = sorted(c[g * gs:(g + 1) * gs], reverse=True)
            gsc.append(vals[0] if gs == 1 else np.float32(vals[0]) + np.float32(vals[1]))
        kept, left = [], list(range(NG))
        for _ in range(tg):
            best = left[0]
            for g in left[1:]:
                if beats(gsc[g], g, gsc[best], best):
                    best = g
            kept.append(best)
            left.remove(best)
        cand = [e for e in range(E) if e // gs in kept]
    else:
        cand = list(range(E))
    picks = []
    for _ in range(K):
        best = cand[0]
        for e in cand[1:]:
            if beats(c[e], e, c[best], best):
                best = e
        picks.append(best)
        cand.remove(best)
    return picks


def chunked(c, K, sig, NG, tg):
    """The kernel's chunked ranking, lane by lane; None where the kernel falls back to
    ranking every allowed expert against every other."""
    E = len(c)
    cl = E // NG if sig else min(E, 32)
    nch, kk = (E + cl - 1) // cl, min(K, cl)
    nkept = tg if sig else nch
    if not (cl <= 32 and nch <= 32 and nch * kk <= 64 and nkept * kk <= 32):
        return None
    ctop, gsc = {}, {}
    for ch in range(nch):  # one warp a chunk, one lane an expert
        base, ln = ch * cl, min(cl, E - ch * cl)
        ranks = [sum(c[base + j] > c[base + l] or (c[base + j] == c[base + l] and j < l) for j in range(ln))
                 for l in range(ln)]
        for l, r in enumerate(ranks):
            if r < kk:
                ctop[ch * kk + r] = base + l
        if sig:
            v0 = c[base + ranks.index(0)]
            gsc[ch] = v0 if ln == 1 else np.float32(v0) + np.float32(c[base + ranks.index(1)])
    if sig:
        kmask = 0
        for g in range(nch):
            if sum(beats(gsc[h], h, gsc[g], g) for h in range(nch)) < tg:
                kmask |= 1 << g
    else:
        kmask = (1 << nch) - 1
    lanes = []
    for lane in range(32):  # one warp a token: lane q * kk + r holds the r-th of kept chunk q
        q, r = divmod(lane, kk)
        mm = kmask
        for _ in range(q):
            mm &= mm - 1
        e = -1
        if lane < nkept * kk and mm:
            ch = (mm & -mm).bit_length() - 1
            if r < min(kk, E - ch * cl):
                e = ctop[ch * kk + r]
        lanes.append(e)
    picks = [None] * K
    for e in lanes:
        if e < 0:
            continue
        rank = sum(beats(c[x], x, c[e], e) for x in lanes if x >= 0)
        if rank < K:
            picks[rank] = e
    return picks


CASES = [  # (E, K, sigmoid, n_group, topk_group)
    (256, 8, True, 8, 4),    # GLM-5.2-shaped
    (64, 8, False, 1, 1),    # OLMoE-shaped (softmax)
    (16, 4, True, 4, 2),     # tiny
    (8, 8, True, 8, 8),      # one expert a group, every expert picked
    (256, 1, True, 8, 1),    # top-1
    (128, 8, True, 4, 2),
    (40, 2, True, 20, 3),
    (96, 3, False, 1, 1),
    (72, 8, False, 1, 1),    # a ragged last run of experts
    (33, 2, False, 1, 1),
]


@pytest.mark.parametrize("E,K,sig,NG,tg", CASES)
def test_chunked_ranking_picks_the_sequential_ids(E, K, sig, NG, tg):
    rng = np.random.default_rng(E * 131 + K)
    for trial in range(24):
        kind = trial % 3
        if kind == 0:
            c = rng.standard_normal(E)
        elif kind == 1:
            c = rng.integers(0, 4, E).astype(np.float64)  # many ties
        else:
            c = rng.standard_normal(E)
            c[rng.integers(0, E, E // 3)] = -np.inf  # NaN scores rank as -inf
        c = [np.float32(x) for x in c]
        got = chunked(c, K, sig, NG, tg)
        assert got is not None
        assert got == sequential(c, K, sig, NG, tg), (trial, got)


def test_fallback_shapes_are_the_ones_the_kernel_ranks_in_full():
    # more than 32 groups, or kept lists wider than a warp: the kernel's full ranking
    assert chunked([np.float32(0)] * 64, 4, True, 64, 4) is None
    assert chunked([np.float32(0)] * 1024, 32, True, 32, 1) is None
