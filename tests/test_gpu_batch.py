"""Many sessions per call: the batched QueryMemory update, rule scores and
top-C* retention against the single-session calls and the oracle, through the
C ABI."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_scores_close, bits, f64

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = kv.Context(0)
    yield c
    c.close()


def _sessions(rng, Ns, n_slots, L, Hq, D, page=16):
    """Per session: a slot map drawn from the shared pool's pages, a unit-norm M, a forced set."""
    out = []
    n_pages = n_slots // page
    for N in Ns:
        pages = rng.choice(n_pages, (N + page - 1) // page, replace=False)
        j = np.arange(N)
        smap = (pages[j // page] * page + j % page).astype(np.int32)
        M = torch.nn.functional.normalize(torch.randn((L, Hq, D), device="cuda"), dim=-1) * float(rng.uniform(1, 6))
        pi = int(rng.integers(0, max(1, N // 8) + 1))
        q_e = N
        q_s = max(pi, N - int(rng.integers(0, max(1, N // 10) + 1)))
        out.append({"N": N, "slot_map": torch.as_tensor(smap, device="cuda"), "M": M, "forced": (min(pi, N), q_s, q_e)})
    return out


@pytest.mark.parametrize("dtype,L,Hq,Hkv,D", [("bf16", 3, 32, 8, 128), ("bf16", 2, 40, 8, 128), ("f32", 2, 8, 4, 64)])
def test_rule_scores_batch_matches_single_calls(ctx, dtype, L, Hq, Hkv, D):
    rng = np.random.default_rng(D + Hq)
    torch.manual_seed(D + Hq)
    n_slots = 48000
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    pool = torch.randn((L, n_slots, Hkv, D), device="cuda").to(tdt)
    Ns = [1, 64, 1000, 5003, 32768, 129]
    sess = _sessions(rng, Ns, n_slots, L, Hq, D)
    rules = [torch.empty(max(N, 1), device="cuda") for N in Ns]
    ctx.rule_scores_batch(pool, [x["M"] for x in sess], L, Hq, Hkv, Ns, D, [x["forced"] for x in sess], rules,
                          slot_maps=[x["slot_map"] for x in sess], n_slots=n_slots)
    ctx.check_device()
    for i, x in enumerate(sess):
        single = torch.empty(max(x["N"], 1), device="cuda")
        pi, qs, qe = x["forced"]
        ctx.rule_scores(pool, x["M"], L, Hq, Hkv, x["N"], D, pi, qs, qe, single, slot_map=x["slot_map"], n_slots=n_slots)
        ctx.check_device()
        assert_scores_close(f64(rules[i][:x["N"]]), f64(single[:x["N"]]), what=f"session {i} vs single call")
    for i in (2, 4):  # two sessions against the oracle
        x = sess[i]
        host_pool = bits(pool).ravel() if dtype == "bf16" else pool.cpu().numpy().ravel()
        ref = oracle.rule_scores(host_pool, x["M"].cpu().double().numpy(), L, Hq, Hkv, x["N"], D, *x["forced"],
                                 slot_map=x["slot_map"].cpu().numpy(), layer_stride=n_slots * Hkv * D)
        assert_scores_close(f64(rules[i][:x["N"]]), ref, what=f"session {i} vs oracle")


def test_rule_scores_batch_full_size(ctx):
    """The batched bench case at full size: 36 sessions of 1024-8192 tokens at the 8B shape
    (L36 Hq32 Hkv8 D128) in one shared paged pool; every session against its single-session
    call, two against the oracle."""
    rng = np.random.default_rng(36)
    torch.manual_seed(36)
    L, Hq, Hkv, D = 36, 32, 8, 128
    Ns = [int(x) for x in rng.integers(1024, 8193, 36)]
    n_slots = sum((x + 15) // 16 for x in Ns) * 16
    pool = torch.randn((L, n_slots, Hkv, D), device="cuda").to(torch.bfloat16)
    perm, at, sess = rng.permutation(n_slots // 16), 0, []
    for N in Ns:
        m = (N + 15) // 16
        j = np.arange(N)
        smap = torch.as_tensor((perm[at:at + m][j // 16] * 16 + j % 16).astype(np.int32), device="cuda")
        at += m
        M = torch.nn.functional.normalize(torch.randn((L, Hq, D), device="cuda"), dim=-1)
        sess.append({"N": N, "slot_map": smap, "M": M, "forced": (64, N - 256, N)})
    rules = [torch.empty(N, device="cuda") for N in Ns]
    ctx.rule_scores_batch(pool, [x["M"] for x in sess], L, Hq, Hkv, Ns, D, [x["forced"] for x in sess], rules,
                          slot_maps=[x["slot_map"] for x in sess], n_slots=n_slots)
    ctx.check_device()
    for i, x in enumerate(sess):
        single = torch.empty(x["N"], device="cuda")
        ctx.rule_scores(pool, x["M"], L, Hq, Hkv, x["N"], D, *x["forced"], single, slot_map=x["slot_map"],
                        n_slots=n_slots)
        assert_scores_close(f64(rules[i]), f64(single), what=f"session {i} vs single call")
    ctx.check_device()
    host_pool = bits(pool).ravel()
    for i in (0, 35):
        x = sess[i]
        ref = oracle.rule_scores(host_pool, x["M"].cpu().double().numpy(), L, Hq, Hkv, x["N"], D, *x["forced"],
                                 slot_map=x["slot_map"].cpu().numpy(), layer_stride=n_slots * Hkv * D)
        assert_scores_close(f64(rules[i]), ref, what=f"session {i} vs oracle")


def test_topk_retain_batch_equals_single_calls(ctx):
    rng = np.random.default_rng(4)
    Ns = [5000, 1, 150000, 32768, 777, 131072]
    Cs = [512, 4, 8192, 100000, 10, 4096]
    rules, forced = [], []
    for N in Ns:
        r = torch.as_tensor(rng.standard_normal(N).astype(np.float32), device="cuda")
        r[: N // 50] = r[0]  # ties
        rules.append(r)
        pi = min(N, 64)
        forced.append((pi, max(pi, N - 128), N))
    keeps = [torch.empty(N, dtype=torch.uint8, device="cuda") for N in Ns]
    idxs = [torch.empty(N, dtype=torch.int32, device="cuda") for N in Ns]
    n_keep = ctx.topk_retain_batch(rules, forced, Cs, keeps, idxs)
    ctx.check_device()
    for i, N in enumerate(Ns):
        k1 = torch.empty(N, dtype=torch.uint8, device="cuda")
        i1 = torch.empty(N, dtype=torch.int32, device="cuda")
        n1 = ctx.topk_retain(rules[i], *forced[i], Cs[i], keep=k1, keep_idx=i1)
        ctx.check_device()
        assert n_keep[i] == n1
        assert torch.equal(keeps[i], k1)
        assert torch.equal(idxs[i][:n1], i1[:n1])
        ref_keep, ref_idx = oracle.topk_retain(rules[i].cpu().double().numpy(), *forced[i], Cs[i])
        assert np.array_equal(keeps[i].cpu().numpy(), ref_keep)


@pytest.mark.parametrize("norm_mode", [0, 1])
def test_memory_update_batch_equals_single_calls(ctx, norm_mode):
    torch.manual_seed(3 + norm_mode)
    L, Hq, D = 4, 32, 128
    Rs, lams, firsts = [256, 16, 1, 100], [0.3, 0.5, 0.0, 2.0], [False, True, False, False]
    qs = [torch.randn((L, Hq, R, D), device="cuda").to(torch.bfloat16) for R in Rs]
    M0 = [torch.nn.functional.normalize(torch.randn((L, Hq, D), device="cuda"), dim=-1) for _ in Rs]
    A0 = [torch.randn((L, Hq, D), device="cuda") for _ in Rs] if norm_mode else None
    Mb = [m.clone() for m in M0]
    Ab = [a.clone() for a in A0] if norm_mode else None
    ctx.memory_update_batch(qs, lams, Mb, first_turn_list=firsts, norm_mode=norm_mode, A_list=Ab)
    ctx.check_device()
    for i in range(len(Rs)):
        M1 = M0[i].clone()
        A1 = A0[i].clone() if norm_mode else None
        ctx.memory_update(qs[i], lams[i], M1, first_turn=firsts[i], norm_mode=norm_mode, A=A1)
        ctx.check_device()
        assert torch.equal(Mb[i], M1)
        if norm_mode:
            assert torch.equal(Ab[i], A1)


def test_batched_token_step(ctx):
    """memory -> rule -> top-C* -> redirect for four sessions in batched calls, against the
    same sessions stepped one by one with the single calls."""
    rng = np.random.default_rng(12)
    torch.manual_seed(12)
    L, Hq, Hkv, D, n_slots = 2, 32, 8, 128, 20000
    pool = torch.randn((L, n_slots, Hkv, D), device="cuda").to(torch.bfloat16)
    Ns, Cs = [4000, 9000, 300, 6000], [1024, 2048, 4096, 512]
    sess = _sessions(rng, Ns, n_slots, L, Hq, D)
    qs = [torch.randn((L, Hq, 64, D), device="cuda").to(torch.bfloat16) for _ in Ns]
    Mb = [x["M"].clone() for x in sess]
    ctx.memory_update_batch(qs, [0.3] * 4, Mb)
    rules = [torch.empty(N, device="cuda") for N in Ns]
    ctx.rule_scores_batch(pool, Mb, L, Hq, Hkv, Ns, D, [x["forced"] for x in sess], rules,
                          slot_maps=[x["slot_map"] for x in sess], n_slots=n_slots)
    keeps = [torch.empty(N, dtype=torch.uint8, device="cuda") for N in Ns]
    ctx.topk_retain_batch(rules, [x["forced"] for x in sess], Cs, keeps)
    ctx.check_device()
    for i, x in enumerate(sess):
        M1 = x["M"].clone()
        ctx.memory_update(qs[i], 0.3, M1)
        assert torch.equal(M1, Mb[i])
        r1 = torch.empty(Ns[i], device="cuda")
        ctx.rule_scores(pool, M1, L, Hq, Hkv, Ns[i], D, *x["forced"], r1, slot_map=x["slot_map"], n_slots=n_slots)
        assert_scores_close(f64(rules[i]), f64(r1), what=f"session {i} rule")
        ref_keep, _ = oracle.topk_retain(f64(rules[i]), *x["forced"], Cs[i])  # on the batched scores
        assert np.array_equal(keeps[i].cpu().numpy(), ref_keep)


@pytest.mark.parametrize("Ns,Cs", [
    # every session fits one CTA (N <= 8192): the batch runs one CTA per session
    ([8192, 1, 2048, 8191, 300, 5000, 8192], [1000, 1, 2048, 20000, 0, 2500, 8191]),
    # sessions up to 16384: one 8-CTA cluster per session
    ([16384, 1, 2048, 16383, 300, 9000, 16384], [1000, 1, 2048, 20000, 0, 4500, 16383]),
])
def test_topk_retain_batch_all_small_sessions(ctx, Ns, Cs):
    """Sessions that fit one launch: one CTA each, or one cluster each."""
    rng = np.random.default_rng(5)
    rules, forced = [], []
    for N in Ns:
        r = np.round(rng.standard_normal(N) * 8) / 8  # many ties
        rules.append(torch.as_tensor(r.astype(np.float32), device="cuda"))
        pi = min(N, 32)
        forced.append((pi, max(pi, N - 64), N))
    keeps = [torch.empty(N, dtype=torch.uint8, device="cuda") for N in Ns]
    idxs = [torch.empty(N, dtype=torch.int32, device="cuda") for N in Ns]
    n_keep = ctx.topk_retain_batch(rules, forced, Cs, keeps, idxs)
    ctx.check_device()
    for i, N in enumerate(Ns):
        ref_keep, ref_idx = oracle.topk_retain(f64(rules[i]), *forced[i], Cs[i])
        assert n_keep[i] == ref_idx.size, f"session {i} (N {N})"
        assert np.array_equal(keeps[i].cpu().numpy(), ref_keep), f"session {i} (N {N})"
        assert np.array_equal(idxs[i][:n_keep[i]].cpu().numpy(), ref_idx), f"session {i} (N {N})"
