"""Pins of the oracle's KVMEM restore path (differential working-set update,
incoming-block restore, in-place position shift) and of SideQuest's
cursor-span eviction mask against what the pages and the mathematics fix:
hand-worked examples, set-partition invariants, degenerate cases, an exact V
copy checked by indexing, the composition law of rotations, and span clearing
re-done with numpy slices.  CPU only."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_fast(rng, shape, scale=1.0):
    x = rng.standard_normal(shape).astype(np.float32) * scale
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f64(bits):
    return oracle.bf16_to_f64(bits)


# --------------------------------------------------------------------------
# differential working-set update
# --------------------------------------------------------------------------

def test_workset_diff_golden():
    g = json.load(open(os.path.join(GOLDEN, "workset_diff_small.json")))
    d = oracle.workset_diff(g["prev_ids"], g["prev_pages"], g["new_ids"], g["P"], g["page"])
    for key in ("new_pages", "shift", "in_rank", "in_page", "mv_rank", "mv_shift", "out_page"):
        assert d[key].tolist() == g[key], key


def _random_sets(rng, universe, n_prev, n_new, P):
    prev = np.sort(rng.choice(universe, n_prev, replace=False)).astype(np.int32)
    new = np.sort(rng.choice(universe, n_new, replace=False)).astype(np.int32)
    pages = rng.choice(P, n_prev, replace=False).astype(np.int32)
    return prev, pages, new


@pytest.mark.parametrize("seed", range(6))
def test_workset_diff_invariants(seed):
    rng = np.random.default_rng(seed)
    universe = int(rng.integers(20, 400))
    n_prev = int(rng.integers(0, min(60, universe)))
    n_new = int(rng.integers(0, min(60, universe)))
    P = max(n_prev, n_new) + int(rng.integers(0, 10))
    page = int(rng.choice([16, 32]))
    prev, pages, new = _random_sets(rng, universe, n_prev, n_new, P)
    d = oracle.workset_diff(prev, pages, new, P, page)
    S_prev, S_new = set(prev.tolist()), set(new.tolist())
    retained = S_prev & S_new
    rank_prev = {b: r for r, b in enumerate(prev.tolist())}
    page_prev = dict(zip(prev.tolist(), pages.tolist()))
    # partition of the new set into retained and incoming
    incoming = {int(new[r]) for r in d["in_rank"]}
    assert incoming == S_new - S_prev
    assert list(d["in_rank"]) == sorted(d["in_rank"])
    # pages: distinct, inside the pool, retained blocks keep theirs
    assert len(set(d["new_pages"].tolist())) == n_new
    assert all(0 <= p < P for p in d["new_pages"])
    for r, b in enumerate(new.tolist()):
        if b in retained:
            assert d["new_pages"][r] == page_prev[b]
            assert d["shift"][r] == (r - rank_prev[b]) * page
        else:
            assert d["shift"][r] == 0
    # incoming pages are the lowest pages not held by a retained block, ascending
    held = {page_prev[b] for b in retained}
    free = [p for p in range(P) if p not in held]
    assert d["in_page"].tolist() == free[:len(incoming)]
    assert [d["new_pages"][r] for r in d["in_rank"]] == d["in_page"].tolist()
    # moved entries: exactly the retained ranks with a non-zero shift
    moved = [r for r, b in enumerate(new.tolist()) if b in retained and r != rank_prev[b]]
    assert d["mv_rank"].tolist() == moved
    assert d["mv_shift"].tolist() == [(r - rank_prev[int(new[r])]) * page for r in moved]
    # outgoing: the previous blocks that left, in ascending block order
    assert d["out_page"].tolist() == [page_prev[b] for b in prev.tolist() if b not in S_new]
    assert len(retained) + len(incoming) == n_new
    assert len(retained) + len(d["out_page"]) == n_prev


def test_workset_diff_degenerate():
    ids = np.array([1, 4, 8], np.int32)
    pages = np.array([2, 0, 1], np.int32)
    same = oracle.workset_diff(ids, pages, ids, 3, 32)
    assert same["new_pages"].tolist() == [2, 0, 1]
    assert same["in_rank"].size == 0 and same["mv_rank"].size == 0 and same["out_page"].size == 0
    disjoint = oracle.workset_diff(ids, pages, np.array([0, 5, 9], np.int32), 3, 32)
    assert disjoint["in_rank"].tolist() == [0, 1, 2]
    assert disjoint["in_page"].tolist() == [0, 1, 2]          # every page is free again
    assert disjoint["out_page"].tolist() == [2, 0, 1]
    first = oracle.workset_diff(np.zeros(0, np.int32), np.zeros(0, np.int32), ids, 5, 32)
    assert first["new_pages"].tolist() == [0, 1, 2] and first["in_rank"].tolist() == [0, 1, 2]
    empty = oracle.workset_diff(ids, pages, np.zeros(0, np.int32), 3, 32)
    assert empty["new_pages"].size == 0 and empty["out_page"].tolist() == [2, 0, 1]
    # an inserted block shifts every later retained block by one page of positions
    shifted = oracle.workset_diff(ids, pages, np.array([0, 1, 4, 8], np.int32), 4, 32)
    assert shifted["mv_rank"].tolist() == [1, 2, 3] and shifted["mv_shift"].tolist() == [32, 32, 32]
    with pytest.raises(ValueError):
        oracle.workset_diff(ids, pages, np.array([0, 1, 4, 8], np.int32), 3, 32)


# --------------------------------------------------------------------------
# incoming-block restore: K re-rotated, V copied
# --------------------------------------------------------------------------

@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_INTERLEAVED])
def test_restore_blocks_v_exact_k_rotation(style):
    rng = np.random.default_rng(7 + style)
    L, Hkv, D, page, nb, P = 2, 3, 16, 4, 5, 6
    k = _bf16_fast(rng, (L, Hkv, nb * page, D))
    v = _bf16_fast(rng, (L, Hkv, nb * page, D))
    src = np.array([3, 0, 4], np.int32)
    dpg = np.array([5, 1, 2], np.int32)
    pos0 = np.array([0, 8, 1000], np.int32)
    kp0 = _bf16_fast(rng, (L, P, page, Hkv, D))
    vp0 = _bf16_fast(rng, (L, P, page, Hkv, D))
    kp, vp = oracle.restore_blocks(k, v, src, dpg, pos0, kp0, vp0, page, 1e4, style)
    untouched = [p for p in range(P) if p not in dpg.tolist()]
    assert np.array_equal(kp[:, untouched], kp0[:, untouched])
    assert np.array_equal(vp[:, untouched], vp0[:, untouched])
    for i in range(src.size):
        rows = slice(src[i] * page, (src[i] + 1) * page)
        # V: the source rows, bit for bit, in [t][g] order
        assert np.array_equal(vp[:, dpg[i]], v[:, :, rows].transpose(0, 2, 1, 3))
        for l in range(L):
            for t in range(page):
                for g in range(Hkv):
                    got = _f64(kp[l, dpg[i], t, g])
                    raw = _f64(k[l, g, src[i] * page + t])
                    pos = pos0[i] + t
                    if pos == 0:
                        assert np.array_equal(got, raw)  # rotation by zero
                    # undoing the rotation gives the raw row back within one bf16 rounding
                    back = oracle.rope_rotate(got, pos, 1e4, style, inverse=True)
                    assert np.allclose(back, raw, rtol=0, atol=2.0 ** -7 * (np.abs(raw).max() + 1e-30))
                    assert abs(np.linalg.norm(got) - np.linalg.norm(raw)) <= 2.0 ** -7 * np.linalg.norm(raw) + 1e-30


# --------------------------------------------------------------------------
# in-place position shift of retained blocks
# --------------------------------------------------------------------------

@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_INTERLEAVED])
def test_rerope_shift_laws(style):
    rng = np.random.default_rng(11 + style)
    L, P, page, Hkv, D = 2, 4, 3, 2, 8
    pool = _bf16_fast(rng, (L, P, page, Hkv, D))
    pages = np.array([1, 3], np.int32)
    zero = oracle.rerope_shift(pool, pages, np.array([0, 0], np.int32), page, 1e6, style)
    assert np.array_equal(zero, pool)                       # shift 0 is the identity, exactly
    fwd = oracle.rerope_shift(pool, pages, np.array([64, -96], np.int32), page, 1e6, style)
    assert np.array_equal(fwd[:, [0, 2]], pool[:, [0, 2]])  # other pages untouched
    back = oracle.rerope_shift(fwd, pages, np.array([-64, 96], np.int32), page, 1e6, style)
    a, b = _f64(back[:, pages]), _f64(pool[:, pages])
    assert np.allclose(a, b, rtol=0, atol=2.0 ** -6 * np.abs(b).max())  # two roundings
    # composition: rotating raw K to p and then shifting by s lands on the rotation to p + s
    raw = rng.standard_normal(D)
    p, s = 37, 1000
    at_p = oracle.bf16_round(oracle.rope_rotate(raw, p, 1e6, style))
    one = np.zeros((1, 1, 1, 1, D), np.uint16)
    one[0, 0, 0, 0] = at_p
    moved = _f64(oracle.rerope_shift(one, np.array([0], np.int32), np.array([s], np.int32), 1, 1e6, style)[0, 0, 0, 0])
    direct = oracle.rope_rotate(raw, p + s, 1e6, style)
    assert np.allclose(moved, direct, rtol=0, atol=2.0 ** -6 * np.abs(direct).max())


# --------------------------------------------------------------------------
# SideQuest cursor-span eviction
# --------------------------------------------------------------------------

def test_span_keep_golden():
    g = json.load(open(os.path.join(GOLDEN, "span_keep_small.json")))
    out, bad = oracle.span_keep(g["span_start"], g["span_end"], g["del_ids"], g["N"], g["keep_in"])
    assert out.tolist() == g["keep_out"] and bad == g["bad_ids"]


@pytest.mark.parametrize("seed", range(5))
def test_span_keep_invariants(seed):
    rng = np.random.default_rng(seed)
    N, n_cur = int(rng.integers(1, 3000)), int(rng.integers(1, 60))
    start = rng.integers(-20, N + 20, n_cur).astype(np.int32)
    end = (start + rng.integers(0, 200, n_cur)).astype(np.int32)
    dels = rng.choice(n_cur + 5, int(rng.integers(0, n_cur)), replace=False).astype(np.int32)
    keep_in = (rng.random(N) < 0.8).astype(np.uint8)
    out, bad = oracle.span_keep(start, end, dels, N, keep_in)
    cleared = np.zeros(N, bool)
    for c in dels:
        if c < n_cur:
            cleared[max(start[c], 0):max(min(end[c], N), 0)] = True
    assert np.array_equal(out.astype(bool), keep_in.astype(bool) & ~cleared)
    assert bad == int((dels >= n_cur).sum())
    # deleting nothing keeps the mask; with no mask given, everything outside the spans is kept
    same, _ = oracle.span_keep(start, end, np.zeros(0, np.int32), N, keep_in)
    assert np.array_equal(same, keep_in)
    ones, _ = oracle.span_keep(start, end, dels, N)
    assert np.array_equal(ones.astype(bool), ~cleared)
    # the deletion order does not matter
    perm, _ = oracle.span_keep(start, end, dels[::-1].copy(), N, keep_in)
    assert np.array_equal(perm, out)
