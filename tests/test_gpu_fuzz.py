"""Seeded randomised parity: shapes, sizes and parameters drawn per seed (ragged tails, odd
group sizes, empty candidate sets, forced sets covering everything, ties) for the calls of
the path, each against the oracle at sizes it finishes in well under a second."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_scores_close, bf16_ulp, bits, f64

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = kv.Context(0)
    yield c
    c.close()


def _bf16(rng, shape, scale=1.0):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("seed", range(24))
def test_block_scores_random_shapes(ctx, seed):
    rng = np.random.default_rng(1000 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.integers(1, 9))
    L, M = int(rng.integers(1, 3)), int(rng.integers(1, 200))
    nb = int(rng.integers(1, 700))
    S = int(rng.integers(0, 6))
    Rc = int(rng.integers(0, 40))
    Bcap = nb + int(rng.integers(0, 5))
    q = _bf16(rng, (L, G * Hkv, M, 128))
    ix = _bf16(rng, (L, Hkv, Bcap, 128), scale=float(rng.uniform(0.1, 1.5)))
    R = torch.empty(nb, device="cuda")
    ctx.block_scores(q, ix, nb, S, Rc, R)
    ctx.check_device()
    ref = oracle.block_scores(bits(q), bits(ix), nb, S, Rc)
    assert_scores_close(f64(R), ref, what=f"R_b seed {seed} (L{L} G{G} Hkv{Hkv} M{M} nb{nb} S{S} R{Rc})")


@pytest.mark.parametrize("seed", range(20))
def test_rule_scores_random_shapes(ctx, seed):
    rng = np.random.default_rng(2000 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 5, 8]))
    L, D = int(rng.integers(1, 4)), int(rng.choice([64, 128]))
    N = int(rng.integers(1, 3000))
    pi = int(rng.integers(0, N + 1))
    q_s = int(rng.integers(pi, N + 1))
    q_e = int(rng.integers(q_s, N + 1))
    paged = bool(rng.integers(0, 2))
    n_slots = N + int(rng.integers(0, 100))
    pool = _bf16(rng, (L, n_slots, Hkv, D))
    M = torch.nn.functional.normalize(torch.from_numpy(rng.standard_normal((L, G * Hkv, D)).astype(np.float32)),
                                      dim=-1).cuda() * float(rng.uniform(1, 8))
    smap = torch.as_tensor(rng.permutation(n_slots)[:N].astype(np.int32), device="cuda") if paged else None
    rule = torch.empty(max(N, 1), device="cuda")
    ctx.rule_scores(pool, M, L, G * Hkv, Hkv, N, D, pi, q_s, q_e, rule, slot_map=smap, n_slots=n_slots)
    ctx.check_device()
    ref = oracle.rule_scores(bits(pool).ravel(), M.cpu().double().numpy(), L, G * Hkv, Hkv, N, D, pi, q_s, q_e,
                             slot_map=None if smap is None else smap.cpu().numpy(), layer_stride=n_slots * Hkv * D)
    assert_scores_close(f64(rule[:N]), ref, what=f"rule seed {seed}")


@pytest.mark.parametrize("seed", range(16))
def test_topk_and_select_random(ctx, seed):
    rng = np.random.default_rng(3000 + seed)
    N = int(rng.integers(1, 200000))
    score = rng.standard_normal(N).astype(np.float32)
    if seed % 3 == 0:
        score = np.round(score * 4) / 4              # many ties
    pi = int(rng.integers(0, min(N, 500) + 1))
    q_s = int(rng.integers(pi, N + 1))
    q_e = int(rng.integers(q_s, min(N, q_s + 300) + 1))
    C = int(rng.integers(0, N + 10))
    s_dev = torch.as_tensor(score, device="cuda")
    keep = torch.empty(N, dtype=torch.uint8, device="cuda")
    idx = torch.empty(N, dtype=torch.int32, device="cuda")
    n = ctx.topk_retain(s_dev, pi, q_s, q_e, C, keep=keep, keep_idx=idx)
    ctx.check_device()
    ref_keep, ref_idx = oracle.topk_retain(score.astype(np.float64), pi, q_s, q_e, C)
    assert n == ref_idx.size
    assert np.array_equal(keep.cpu().numpy(), ref_keep)
    assert np.array_equal(idx[:n].cpu().numpy(), ref_idx)
    # working-set selection on the same scores, as block relevance
    n_sink, n_recent = int(rng.integers(0, 5)), int(rng.integers(0, 50))
    k = int(rng.integers(0, N + 5))
    R = np.abs(score).astype(np.float32)
    ids = torch.empty(N, dtype=torch.int32, device="cuda")
    ns = ctx.select_blocks(torch.as_tensor(R, device="cuda"), n_sink, n_recent, k, ids)
    ctx.check_device()
    ref_ids = oracle.select_blocks(R.astype(np.float64), n_sink, n_recent, k)
    assert ns == ref_ids.size and np.array_equal(ids[:ns].cpu().numpy(), ref_ids)


@pytest.mark.parametrize("seed", range(10))
def test_meank_random_shapes(ctx, seed):
    rng = np.random.default_rng(4000 + seed)
    L, Hkv = int(rng.integers(1, 3)), int(rng.choice([1, 2, 8]))
    D = int(rng.choice([64, 128, 256]))
    block = int(rng.choice([8, 16, 32, 64]))
    T = int(rng.integers(1, 40 * block))
    k = _bf16(rng, (L, Hkv, T, D))
    nb = (T + block - 1) // block
    Bcap = nb + int(rng.integers(0, 3))
    index = torch.zeros((L, Hkv, Bcap, D), dtype=torch.bfloat16, device="cuda")
    ctx.meank_build(k, block, index)
    ctx.check_device()
    ref = oracle.meank_build(bits(k), block, Bcap=Bcap)
    got, want = oracle.bf16_to_f64(bits(index)), oracle.bf16_to_f64(ref)
    bad = np.flatnonzero(np.abs(got - want) > bf16_ulp(want) * (1 + 1e-12))
    assert bad.size == 0, f"Mean-K seed {seed} (T{T} block{block} D{D}): {bad.size} beyond 1 ulp"
    assert np.array_equal(bits(index)[:, :, nb:], ref[:, :, nb:])   # capacity past the blocks untouched


@pytest.mark.parametrize("seed", range(8))
def test_fp8_index_random(ctx, seed):
    rng = np.random.default_rng(5000 + seed)
    D = int(rng.choice([64, 128, 256]))
    rows = int(rng.integers(1, 5000))
    x = rng.standard_normal((rows, D)) * 10.0 ** rng.uniform(-30, 30, (rows, 1))
    x[rng.random(rows) < 0.05] = 0.0
    idx = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).cuda()
    codes, exps = ctx.index_to_fp8(idx)
    back = ctx.index_from_fp8(codes, exps)
    ctx.check_device()
    rc, re_ = oracle.index_to_fp8(bits(idx))
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(exps.cpu().numpy(), re_)
    assert np.array_equal(bits(back), oracle.index_from_fp8(rc, re_))


@pytest.mark.parametrize("seed", range(8))
def test_topk_batch_random_sessions(ctx, seed):
    rng = np.random.default_rng(6000 + seed)
    S = int(rng.integers(1, 13))
    Ns = [int(rng.choice([rng.integers(1, 2000), rng.integers(2000, 140000), rng.integers(131073, 300000)]))
          for _ in range(S)]
    rules, forced, Cs = [], [], []
    for N in Ns:
        r = rng.standard_normal(N).astype(np.float32)
        if rng.integers(0, 2):
            r = np.round(r * 8) / 8
        rules.append(torch.as_tensor(r, device="cuda"))
        pi = int(rng.integers(0, min(N, 300) + 1))
        q_s = int(rng.integers(pi, N + 1))
        forced.append((pi, q_s, int(rng.integers(q_s, min(N, q_s + 500) + 1))))
        Cs.append(int(rng.integers(0, N + 3)))
    keeps = [torch.empty(N, dtype=torch.uint8, device="cuda") for N in Ns]
    idxs = [torch.empty(N, dtype=torch.int32, device="cuda") for N in Ns]
    n_keep = ctx.topk_retain_batch(rules, forced, Cs, keeps, idxs)
    ctx.check_device()
    for i in range(S):
        ref_keep, ref_idx = oracle.topk_retain(f64(rules[i]), *forced[i], Cs[i])
        assert n_keep[i] == ref_idx.size, f"session {i} of {S} (N {Ns[i]})"
        assert np.array_equal(keeps[i].cpu().numpy(), ref_keep), f"session {i} of {S} (N {Ns[i]})"
        assert np.array_equal(idxs[i][:n_keep[i]].cpu().numpy(), ref_idx), f"session {i} of {S}"


@pytest.mark.parametrize("seed", range(8))
def test_span_keep_random(ctx, seed):
    rng = np.random.default_rng(7000 + seed)
    N = int(rng.integers(1, 100000))
    n_cur = int(rng.integers(0, 60))
    starts = rng.integers(-100, N + 100, n_cur).astype(np.int32)       # spans may overlap and run past [0, N)
    ends = (starts + rng.integers(0, 4000, n_cur)).astype(np.int32)
    dels = rng.permutation(n_cur)[:int(rng.integers(0, n_cur + 1))].astype(np.int32)
    keep_in = (rng.random(N) < 0.7).astype(np.uint8)
    out = torch.empty(N, dtype=torch.uint8, device="cuda")
    ctx.span_keep(torch.as_tensor(starts, device="cuda"), torch.as_tensor(ends, device="cuda"),
                  torch.as_tensor(dels, device="cuda"), N, out, keep_in=torch.as_tensor(keep_in, device="cuda"))
    ctx.check_device()
    ref, n_bad = oracle.span_keep(starts, ends, dels, N, keep_in=keep_in)
    assert n_bad == 0 and np.array_equal(out.cpu().numpy(), ref)
