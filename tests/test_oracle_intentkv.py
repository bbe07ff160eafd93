"""Pins of the fp64 oracle's IntentKV half (QueryMemory, rule scores, top-C*
retention, dead-slot redirect) against what the page and the mathematics fix:
hand-worked examples (tests/golden), closed forms, invariants, library
special cases and brute force.  CPU only."""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

import oracle


# --------------------------------------------------------------------------
# QueryMemory (IntentKV Sec. 3.2, Eq. 2)
# --------------------------------------------------------------------------

def _turns(rng, T, L, Hq, R, D):
    return [rng.standard_normal((L, Hq, R, D)).astype(np.float32) for _ in range(T)]


def test_memory_golden_two_turns(golden):
    g = golden("memory_update_two_turns.json")
    t1 = np.array(g["turns"][0], dtype=np.float32)[None, None]
    t2 = np.array(g["turns"][1], dtype=np.float32)[None, None]
    M1, _ = oracle.memory_update(t1, g["lambda"], first_turn=True)
    np.testing.assert_allclose(M1[0, 0], g["M1"], atol=1e-15)
    M2, _ = oracle.memory_update(t2, g["lambda"], M=M1)
    np.testing.assert_allclose(M2[0, 0], g["M2_mode0"], rtol=1e-14)
    M1b, A1 = oracle.memory_update(t1, g["lambda"], first_turn=True, norm_mode=1)
    M2b, A2 = oracle.memory_update(t2, g["lambda"], M=M1b, A=A1, norm_mode=1)
    np.testing.assert_allclose(A2[0, 0], g["A2_mode1"], rtol=1e-14)
    np.testing.assert_allclose(M2b[0, 0], g["M2_mode1"], rtol=1e-14)


@pytest.mark.parametrize("norm_mode", [0, 1])
def test_memory_unit_norm(norm_mode):
    rng = np.random.default_rng(1)
    M = A = None
    for t, q in enumerate(_turns(rng, 4, 2, 3, 5, 16)):
        M, A = oracle.memory_update(q, 0.4, M=M, A=A, first_turn=(t == 0), norm_mode=norm_mode)
        np.testing.assert_allclose(np.linalg.norm(M, axis=-1), 1.0, atol=1e-12)


def test_memory_first_turn_is_normalised_mean():
    rng = np.random.default_rng(2)
    q = _turns(rng, 1, 2, 2, 7, 8)[0]
    garbage = rng.standard_normal((2, 2, 8))  # previous state must be ignored
    M, _ = oracle.memory_update(q, 0.3, M=garbage, first_turn=True)
    E = q.astype(np.float64).mean(axis=2)
    np.testing.assert_allclose(M, E / np.linalg.norm(E, axis=-1, keepdims=True), rtol=1e-13)


def test_memory_mode1_closed_form():
    """norm_mode 1 carries A_t = sum_s e^{-lam (t-s)} E_s (geometric sum)."""
    rng = np.random.default_rng(3)
    lam = 0.7
    qs = _turns(rng, 5, 1, 2, 3, 8)
    M = A = None
    for t, q in enumerate(qs):
        M, A = oracle.memory_update(q, lam, M=M, A=A, first_turn=(t == 0), norm_mode=1)
    T = len(qs)
    E = [q.astype(np.float64).mean(axis=2) for q in qs]
    Acf = sum(np.exp(-lam * (T - 1 - s)) * E[s] for s in range(T))
    np.testing.assert_allclose(A, Acf, rtol=1e-12)
    np.testing.assert_allclose(M, Acf / np.linalg.norm(Acf, axis=-1, keepdims=True), rtol=1e-12)


def test_memory_mode0_unrolled_closed_form():
    """Unrolled: U_t = sum_s e^{-lam (t-s)} E_s / prod_{r=s}^{t-1} n_r, n_r = |U_r|, M_t = U_t / n_t."""
    rng = np.random.default_rng(4)
    lam = 0.25
    qs = _turns(rng, 6, 2, 1, 4, 8)
    E = [q.astype(np.float64).mean(axis=2) for q in qs]
    norms = []
    M = None
    for t, q in enumerate(qs):
        M, _ = oracle.memory_update(q, lam, M=M, first_turn=(t == 0))
        U = np.zeros_like(E[0])
        for s in range(t + 1):
            denom = np.ones_like(norms[0]) if norms else 1.0
            for r in range(s, t):
                denom = denom * norms[r]
            U = U + np.exp(-lam * (t - s)) * E[s] / denom
        n_t = np.linalg.norm(U, axis=-1, keepdims=True)
        norms.append(n_t)
        np.testing.assert_allclose(M, U / n_t, rtol=1e-11)


def test_memory_fixed_point_and_query_mode():
    rng = np.random.default_rng(5)
    q = _turns(rng, 1, 1, 2, 3, 8)[0]
    E = q.astype(np.float64).mean(axis=2)
    target = E / np.linalg.norm(E, axis=-1, keepdims=True)
    M = None
    for t in range(5):  # the same span every turn: M stays E/|E|
        M, _ = oracle.memory_update(q, 0.3, M=M, first_turn=(t == 0))
        np.testing.assert_allclose(M, target, rtol=1e-13)
    # lambda -> infinity forgets the past entirely: query mode, M = E_t/|E_t|
    q2 = _turns(rng, 1, 1, 2, 3, 8)[0]
    M2, _ = oracle.memory_update(q2, 1e4, M=M)
    E2 = q2.astype(np.float64).mean(axis=2)
    np.testing.assert_allclose(M2, E2 / np.linalg.norm(E2, axis=-1, keepdims=True), rtol=1e-13)


def test_memory_decay_sign():
    """e^{-lambda} shrinks the past: with a large lambda the newest turn dominates."""
    old = np.zeros((1, 1, 1, 2), np.float32); old[..., 0] = 1
    new = np.zeros((1, 1, 1, 2), np.float32); new[..., 1] = 1
    M, _ = oracle.memory_update(old, 3.0, first_turn=True)
    M, _ = oracle.memory_update(new, 3.0, M=M)
    assert M[0, 0, 1] > 0.99 and abs(M[0, 0, 0] - np.exp(-3.0) / np.hypot(np.exp(-3.0), 1)) < 1e-15


def test_memory_zero_and_bf16():
    z = np.zeros((1, 1, 4, 8), np.float32)
    M, _ = oracle.memory_update(z, 0.5, first_turn=True)
    assert np.all(M == 0)
    rng = np.random.default_rng(6)
    q = rng.standard_normal((2, 2, 3, 8)).astype(np.float32)
    bits = oracle.bf16_round(q)  # bf16 input path widens exactly
    Mb, _ = oracle.memory_update(bits, 0.5, first_turn=True)
    Mf, _ = oracle.memory_update(oracle.bf16_to_f64(bits).astype(np.float32), 0.5, first_turn=True)
    np.testing.assert_array_equal(Mb, Mf)


# --------------------------------------------------------------------------
# rule scores (IntentKV Sec. 3.2, Eq. 3-4)
# --------------------------------------------------------------------------

def _unit(rng, *shape):
    m = rng.standard_normal(shape)
    return m / np.linalg.norm(m, axis=-1, keepdims=True)


def test_rule_golden(golden):
    g = golden("rule_scores_tiny.json")
    K = np.array(g["K"], np.float32)  # [N, D] -> pool [L=1][N][Hkv=1][D]
    rule = oracle.rule_scores(K, np.array(g["M"]), g["L"], g["Hq"], g["Hkv"], g["N"], g["D"],
                              g["pi"], g["q_s"], g["q_e"])
    np.testing.assert_allclose(rule, g["rule"], rtol=1e-6, atol=1e-7)


def _rand_pool(rng, L, N, Hkv, D):
    return rng.standard_normal((L, N, Hkv, D)).astype(np.float32)


def test_rule_sum_and_forced_zero():
    rng = np.random.default_rng(10)
    L, Hq, Hkv, N, D = 3, 6, 2, 100, 16
    K = _rand_pool(rng, L, N, Hkv, D)
    M = _unit(rng, L, Hq, D)
    pi, qs, qe = 7, 80, 95
    rule = oracle.rule_scores(K, M, L, Hq, Hkv, N, D, pi, qs, qe)
    assert abs(rule.sum() - L * Hq) < 1e-9
    F = np.r_[0:pi, qs:qe]
    assert np.all(rule[F] == 0)
    assert np.all(rule[np.setdiff1d(np.arange(N), F)] > 0)


def test_rule_constant_k_uniform():
    rng = np.random.default_rng(11)
    L, Hq, Hkv, N, D = 2, 4, 2, 50, 8
    K = np.broadcast_to(rng.standard_normal((1, 1, Hkv, D)), (L, N, Hkv, D)).astype(np.float32)
    M = _unit(rng, L, Hq, D)
    rule = oracle.rule_scores(K.copy(), M, L, Hq, Hkv, N, D, 5, 45, 50)
    nH = N - 10
    np.testing.assert_allclose(rule[5:45], L * Hq / nH, rtol=1e-13)


def test_rule_library_softmax_brute_force():
    rng = np.random.default_rng(12)
    L, Hq, Hkv, N, D = 2, 6, 3, 37, 8
    K = _rand_pool(rng, L, N, Hkv, D)
    M = _unit(rng, L, Hq, D) * 3.0
    pi, qs, qe = 3, 30, 34
    rule = oracle.rule_scores(K, M, L, Hq, Hkv, N, D, pi, qs, qe)
    H = np.array([j for j in range(N) if not (j < pi or qs <= j < qe)])
    G = Hq // Hkv
    ref = np.zeros(N)
    for l in range(L):
        for h in range(Hq):
            logits = K[l, H, h // G, :].astype(np.float64) @ M[l, h] / np.sqrt(D)
            ref[H] += softmax(logits)
    np.testing.assert_allclose(rule, ref, rtol=1e-12, atol=1e-15)


def test_rule_gqa_contiguous_groups():
    """Heads 0,1 read kv head 0 and heads 2,3 read kv head 1 (contiguous grouping)."""
    L, Hq, Hkv, N, D = 1, 4, 2, 20, 4
    K = np.zeros((L, N, Hkv, D), np.float32)
    K[0, 5, 0, 0] = 40.0   # kv head 0: spike along e0 at j=5
    K[0, 9, 1, 1] = 40.0   # kv head 1: spike along e1 at j=9
    M = np.zeros((L, Hq, D))
    M[0, 0:2, 0] = 1.0     # heads of group 0 look along e0
    M[0, 2:4, 1] = 1.0     # heads of group 1 look along e1
    rule = oracle.rule_scores(K, M, L, Hq, Hkv, N, D, 0, N, N)
    assert rule[5] > 1.99 and rule[9] > 1.99


def test_rule_scale_is_sqrt_d():
    """Two candidates with logits 0 and x/sqrt(D): a missing or wrong scale changes the split."""
    D = 16
    K = np.zeros((1, 2, 1, D), np.float32)
    K[0, 1, 0, 0] = 8.0
    M = np.zeros((1, 1, D)); M[0, 0, 0] = 1.0
    rule = oracle.rule_scores(K, M, 1, 1, 1, 2, D, 0, 2, 2)
    p = np.exp(2.0) / (1 + np.exp(2.0))  # 8 / sqrt(16) = 2
    np.testing.assert_allclose(rule, [1 - p, p], rtol=1e-14)


def test_rule_slot_map_and_strides():
    """Reading through a paged slot map equals reading the gathered dense K."""
    rng = np.random.default_rng(13)
    L, Hq, Hkv, N, D, page = 2, 4, 2, 64, 8, 16
    slots = N + 16  # pool larger than N, padded rows
    pool = rng.standard_normal((L, slots, Hkv, D + 8)).astype(np.float32)  # slot stride != Hkv*D
    perm = rng.permutation(slots // page)
    smap = np.array([perm[j // page] * page + j % page for j in range(N)], np.int32)
    M = _unit(rng, L, Hq, D)
    flat = pool.ravel()
    slot_stride = Hkv * (D + 8)
    # heads inside a slot are D apart: lay the D+8-wide rows out so head g starts at g*D
    rule = oracle.rule_scores(flat, M, L, Hq, Hkv, N, D, 4, 60, 64, slot_map=smap,
                              layer_stride=slots * slot_stride, slot_stride=slot_stride)
    rows = flat.reshape(L, slots, slot_stride)
    dense = np.stack([rows[:, smap[j], :Hkv * D] for j in range(N)], axis=1).reshape(L, N, Hkv, D)
    ref = oracle.rule_scores(np.ascontiguousarray(dense), M, L, Hq, Hkv, N, D, 4, 60, 64)
    np.testing.assert_array_equal(rule, ref)


def test_rule_permutation_equivariance():
    rng = np.random.default_rng(14)
    L, Hq, Hkv, N, D = 2, 2, 1, 30, 8
    K = _rand_pool(rng, L, N, Hkv, D)
    M = _unit(rng, L, Hq, D)
    pi = 4
    rule = oracle.rule_scores(K, M, L, Hq, Hkv, N, D, pi, N, N)
    perm = np.r_[np.arange(pi), pi + rng.permutation(N - pi)]
    rule_p = oracle.rule_scores(np.ascontiguousarray(K[:, perm]), M, L, Hq, Hkv, N, D, pi, N, N)
    np.testing.assert_allclose(rule_p, rule[perm], rtol=1e-12)


def test_rule_dominant_position_and_empty_h():
    rng = np.random.default_rng(15)
    L, Hq, Hkv, N, D = 1, 2, 1, 40, 8
    K = (0.01 * rng.standard_normal((L, N, Hkv, D))).astype(np.float32)
    M = _unit(rng, L, Hq, D)
    K[0, 17, 0] = (200.0 * M[0, 0]).astype(np.float32) + (200.0 * M[0, 1]).astype(np.float32)
    rule = oracle.rule_scores(K, M, L, Hq, Hkv, N, D, 0, N, N)
    assert rule[17] > L * Hq - 1e-6
    empty = oracle.rule_scores(K, M, L, Hq, Hkv, N, D, 20, 20, N)  # F covers everything
    assert np.all(empty == 0)


# --------------------------------------------------------------------------
# top-C* retention (IntentKV Sec. 3.1, Eq. 1)
# --------------------------------------------------------------------------

def test_topk_golden(golden):
    g = golden("topk_retain_tiny.json")
    keep, idx = oracle.topk_retain(np.array(g["score"]), g["pi"], g["q_s"], g["q_e"], g["C"])
    assert idx.tolist() == g["keep_idx"]
    assert keep.sum() == len(g["keep_idx"])


@pytest.mark.parametrize("seed", range(6))
def test_topk_invariants_and_sort(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 300))
    pi = int(rng.integers(0, N + 1))
    qs = int(rng.integers(0, N + 1)); qe = int(rng.integers(qs, N + 1))
    C = int(rng.integers(0, N + 5))
    s = np.round(rng.random(N), 2)  # many exact ties
    keep, idx = oracle.topk_retain(s, pi, qs, qe, C)
    F = set(range(pi)) | set(range(qs, qe))
    H = [j for j in range(N) if j not in F]
    cstar = max(0, C - len(F))
    assert F <= set(idx.tolist())
    assert len(idx) == len(F) + min(cstar, len(H))
    assert np.all(np.diff(idx) > 0) and keep.sum() == len(idx)
    kept = [j for j in H if keep[j]]
    dropped = [j for j in H if not keep[j]]
    if kept and dropped:
        assert min(s[kept]) >= max(s[dropped])
    ref = sorted(H, key=lambda j: (-s[j], j))[:cstar]
    assert sorted(ref) == kept
    if N <= C:
        assert keep.all()


@pytest.mark.parametrize("seed", range(4))
def test_topk_exhaustive_subset(seed):
    """Eq. 1 as written: the C*-subset of H with the largest score sum (distinct scores)."""
    rng = np.random.default_rng(100 + seed)
    N = 11
    s = rng.permutation(N).astype(np.float64) + rng.random()
    pi, qs, qe, C = 2, 9, 10, 6
    keep, idx = oracle.topk_retain(s, pi, qs, qe, C)
    H = [j for j in range(N) if not (j < pi or qs <= j < qe)]
    cstar = C - 3
    best = max(itertools.combinations(H, cstar), key=lambda sub: sum(s[list(sub)]))
    assert sorted(set(idx.tolist()) - {0, 1, 9}) == sorted(best)


def test_topk_nan_and_signed_zero():
    s = np.array([np.nan, 0.0, -0.0, 0.5, np.nan, -1.0])
    keep, idx = oracle.topk_retain(s, 0, 6, 6, 3)
    assert idx.tolist() == [1, 2, 3]   # NaN ranks lowest; -0 ties +0, lower index first
    keep, idx = oracle.topk_retain(s, 0, 6, 6, 5)
    assert idx.tolist() == [0, 1, 2, 3, 5]


# --------------------------------------------------------------------------
# dead-slot redirect (IntentKV abstract and Sec. 3: layout layer)
# --------------------------------------------------------------------------

def test_redirect_pins():
    rng = np.random.default_rng(20)
    N = 200
    slot_in = rng.permutation(N).astype(np.int32)
    keep = (rng.random(N) < 0.3).astype(np.uint8)
    out = oracle.redirect_slots(slot_in, keep, N)
    assert np.array_equal(out[keep == 1], slot_in[keep == 1])     # survivors never move
    assert np.all(out[keep == 0] == N)                            # dropped -> dead slot
    assert (out == N).sum() == N - keep.sum()
    assert np.array_equal(oracle.redirect_slots(out, keep, N), out)  # idempotent
