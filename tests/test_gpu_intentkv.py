"""Parity of the CUDA IntentKV path (QueryMemory, rule scores, top-C*, dead-slot
redirect) with the fp64 oracle, through the C ABI, on seeded synthetic inputs."""
import numpy as np
import pytest
import torch

import oracle
from helpers import (assert_keep_sets_match, assert_scores_close, bits, f64)

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402
import synth  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = kv.Context(0)
    yield c
    c.close()


def _host(t):
    """Oracle-side copy of an input tensor: bf16 -> uint16 bits, fp32 -> float32."""
    return bits(t) if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


def _oracle_memory(w, turns):
    M = A = None
    for t in range(w.turns):
        M, A = oracle.memory_update(_host(turns[t]), w.lam, M=M, first_turn=(t == 0))
    return M


def _gpu_memory(ctx, w, turns, norm_mode=0):
    M = torch.zeros((w.L, w.Hq, w.D), device="cuda")
    A = torch.zeros_like(M) if norm_mode else None
    for t in range(w.turns):
        ctx.memory_update(turns[t], w.lam, M, first_turn=(t == 0), norm_mode=norm_mode, A=A)
    return M


def _forced(w):
    return lambda j: j < w.pi or (w.q_s <= j < w.q_e)


# ---------------------------------------------------------------------------
# QueryMemory
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "8b", "long"])
def test_memory_update_parity(ctx, name):
    w = synth.TOKEN[name]
    turns = synth.token_inputs(w, "cuda")["turns"]
    M_gpu = _gpu_memory(ctx, w, turns)
    torch.cuda.synchronize()
    M_ref = _oracle_memory(w, turns)
    assert_scores_close(f64(M_gpu), M_ref, what="M_t")
    np.testing.assert_allclose(np.linalg.norm(f64(M_gpu), axis=-1), 1.0, atol=1e-5)


def test_memory_update_mode1_and_zero(ctx):
    w = synth.scaled(synth.TOKEN["tiny"], turns=4)
    turns = synth.token_inputs(w, "cuda")["turns"]
    turns[2, 0, 1] = 0  # one head with a zero span in turn 2 only
    M_gpu = _gpu_memory(ctx, w, turns, norm_mode=1)
    M = A = None
    for t in range(w.turns):
        M, A = oracle.memory_update(_host(turns[t]), w.lam, M=M, A=A, first_turn=(t == 0), norm_mode=1)
    assert_scores_close(f64(M_gpu), M, what="M_t mode 1")
    z = torch.zeros((1, 1, 5, 64), device="cuda")
    Mz = torch.full((1, 1, 64), 7.0, device="cuda")
    ctx.memory_update(z, 0.5, Mz, first_turn=True)
    assert torch.all(Mz == 0)


def test_query_mode_ignores_the_session_memory(ctx):
    """IntentKV's query mode scores with the current query encoding alone: an update with
    first_turn set gives Enc(q_t)/|Enc(q_t)| whatever the session's memory held."""
    w = synth.TOKEN["8b"]
    turns = synth.token_inputs(synth.scaled(w, L=2, N=64, turns=2), "cuda")["turns"]
    fresh = torch.zeros((2, w.Hq, w.D), device="cuda")
    used = torch.randn((2, w.Hq, w.D), device="cuda")
    ctx.memory_update(turns[1], w.lam, fresh, first_turn=True)
    ctx.memory_update(turns[1], w.lam, used, first_turn=True)
    assert torch.equal(fresh, used)
    ref, _ = oracle.memory_update(_host(turns[1]), w.lam, first_turn=True)
    assert_scores_close(f64(fresh), ref, what="query-mode M")
    assert torch.allclose(fresh.norm(dim=-1), torch.ones(2, w.Hq, device="cuda"), atol=1e-5)


def test_memory_update_ragged_dims(ctx):
    # D=72 (not a power of two), R=3, bf16 rows
    g = torch.Generator(device="cuda").manual_seed(7)
    q = torch.randn((3, 5, 3, 72), generator=g, device="cuda").to(torch.bfloat16)
    M = torch.randn((3, 5, 72), generator=g, device="cuda")
    M0 = M.detach().cpu().double().numpy()
    ctx.memory_update(q, 0.8, M)
    ref, _ = oracle.memory_update(bits(q), 0.8, M=M0)
    assert_scores_close(f64(M), ref, what="M_t D=72")


@pytest.mark.parametrize("dtype,D,R", [(torch.bfloat16, 1024, 300), (torch.float32, 1024, 77), (torch.float32, 520, 5),
                                       (torch.bfloat16, 16, 1000)])
def test_memory_update_wide_and_narrow_rows(ctx, dtype, D, R):
    """Rows of up to 1024 dims (one thread per 16-byte chunk, one row per pass) and of 16 dims
    (64 rows per pass)."""
    g = torch.Generator(device="cuda").manual_seed(D + R)
    q = torch.randn((2, 3, R, D), generator=g, device="cuda").to(dtype)
    M = torch.randn((2, 3, D), generator=g, device="cuda")
    M0 = M.detach().cpu().double().numpy()
    ctx.memory_update(q, 0.3, M)
    qh = bits(q) if dtype == torch.bfloat16 else q.cpu().numpy()
    ref, _ = oracle.memory_update(qh, 0.3, M=M0)
    assert_scores_close(f64(M), ref, what=f"M_t D={D} R={R}")


# ---------------------------------------------------------------------------
# rule scores
# ---------------------------------------------------------------------------

def _rule_pair(ctx, w, inp, M32):
    """GPU and oracle rule scores on the same inputs (M given as fp32)."""
    rule = torch.empty(w.N, device="cuda")
    ctx.rule_scores(inp["pool"], M32, w.L, w.Hq, w.Hkv, w.N, w.D, w.pi, w.q_s, w.q_e, rule,
                    slot_map=inp["slot_map"], n_slots=w.N)
    torch.cuda.synchronize()
    sm = None if inp["slot_map"] is None else inp["slot_map"].cpu().numpy()
    ref = oracle.rule_scores(_host(inp["pool"]).ravel(), M32.cpu().double().numpy(), w.L, w.Hq, w.Hkv, w.N, w.D,
                             w.pi, w.q_s, w.q_e, slot_map=sm)
    return f64(rule), ref


@pytest.mark.parametrize("name", ["tiny", "8b", "long"])
def test_rule_scores_parity_full_size(ctx, name):
    w = synth.TOKEN[name]
    inp = synth.token_inputs(w, "cuda")
    M32 = torch.from_numpy(_oracle_memory(w, inp["turns"]).astype(np.float32)).cuda()
    got, ref = _rule_pair(ctx, w, inp, M32)
    assert_scores_close(got, ref, what=f"rule_j ({name})")
    assert abs(got.sum() - w.L * w.Hq) < 1e-3 * w.L * w.Hq
    F = np.r_[0:w.pi, w.q_s:w.q_e]
    assert np.all(got[F] == 0)
    ctx.check_device()


@pytest.mark.parametrize("Hq", [10, 8])  # G = 5 and G = 4
@pytest.mark.parametrize("N,pi,qs,qe", [(1000, 3, 950, 1000), (129, 0, 129, 129), (64, 10, 20, 30),
                                        (1, 0, 1, 1), (300, 300, 300, 300), (77, 76, 0, 1)])
def test_rule_scores_ragged_and_degenerate(ctx, N, pi, qs, qe, Hq):
    w = synth.scaled(synth.TOKEN["8b"], L=2, Hq=Hq, Hkv=2, N=N, turns=1, R=4, page=0)
    inp = synth.token_inputs(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(N)
    M32 = torch.nn.functional.normalize(torch.randn((w.L, w.Hq, w.D), generator=g, device="cuda"), dim=-1)
    rule = torch.empty(N, device="cuda")
    ctx.rule_scores(inp["pool"], M32, w.L, w.Hq, w.Hkv, N, w.D, pi, qs, qe, rule, n_slots=N)
    ref = oracle.rule_scores(bits(inp["pool"]).ravel(), M32.cpu().double().numpy(), w.L, w.Hq, w.Hkv, N, w.D, pi, qs,
                             qe)
    assert_scores_close(f64(rule), ref, what="rule_j degenerate")


@pytest.mark.parametrize("G,Hkv,D", [(1, 4, 64), (3, 2, 128), (5, 1, 256), (8, 2, 32), (2, 3, 16),
                                     (1, 8, 128), (2, 4, 128), (4, 8, 128), (5, 8, 128), (6, 2, 128),
                                     (7, 1, 128), (8, 16, 128), (4, 16, 128)])
def test_rule_scores_shapes(ctx, G, Hkv, D):
    L, N = 2, 333
    Hq = G * Hkv
    gen = torch.Generator(device="cuda").manual_seed(G * 100 + D)
    pool = torch.randn((L, N + 7, Hkv, D), generator=gen, device="cuda").to(torch.bfloat16)
    smap = torch.randperm(N + 7, generator=gen, device="cuda")[:N].to(torch.int32)
    M32 = torch.nn.functional.normalize(torch.randn((L, Hq, D), generator=gen, device="cuda"), dim=-1) * 4
    rule = torch.empty(N, device="cuda")
    ctx.rule_scores(pool, M32, L, Hq, Hkv, N, D, 5, 300, 320, rule, slot_map=smap, n_slots=N + 7)
    ref = oracle.rule_scores(bits(pool).ravel(), M32.cpu().double().numpy(), L, Hq, Hkv, N, D, 5, 300, 320,
                             slot_map=smap.cpu().numpy(), slot_stride=Hkv * D, layer_stride=(N + 7) * Hkv * D)
    assert_scores_close(f64(rule), ref, what=f"rule_j G={G} Hkv={Hkv} D={D}")


@pytest.mark.parametrize("D", [64, 128])
def test_rule_scores_strided_pool_16B_aligned(ctx, D):
    """slot_stride with 16-byte (not 32-byte) alignment takes the split-load path."""
    L, Hq, Hkv, N = 2, 4, 2, 200
    stride = Hkv * D + 8  # 16 bytes of padding per slot in bf16
    gen = torch.Generator(device="cuda").manual_seed(3)
    flat = torch.randn((L, N, stride), generator=gen, device="cuda").to(torch.bfloat16)
    M32 = torch.nn.functional.normalize(torch.randn((L, Hq, D), generator=gen, device="cuda"), dim=-1)
    rule = torch.empty(N, device="cuda")
    ctx.rule_scores(flat, M32, L, Hq, Hkv, N, D, 2, 190, 200, rule, n_slots=N, slot_stride=stride,
                    layer_stride=N * stride)
    ref = oracle.rule_scores(bits(flat).ravel(), M32.cpu().double().numpy(), L, Hq, Hkv, N, D, 2, 190, 200,
                             slot_stride=stride, layer_stride=N * stride)
    assert_scores_close(f64(rule), ref, what="rule_j strided")


@pytest.mark.parametrize("Hq,D", [(2, 64), (4, 128)])
def test_rule_scores_bad_slot_sets_device_error(ctx, Hq, D):
    L, Hkv, N = 1, 1, 40
    pool = torch.zeros((L, N, Hkv, D), device="cuda", dtype=torch.bfloat16)
    smap = torch.arange(N, device="cuda", dtype=torch.int32)
    smap[17] = N + 5  # outside the pool: read as a zero row and flagged
    M32 = torch.nn.functional.normalize(torch.ones((L, Hq, D), device="cuda"), dim=-1)
    rule = torch.empty(N, device="cuda")
    ctx.rule_scores(pool, M32, L, Hq, Hkv, N, D, 0, N, N, rule, slot_map=smap, n_slots=N)
    with pytest.raises(kv.KvselError) as e:
        ctx.check_device()
    assert e.value.code == kv.ERR_DEVICE_CHECK
    ctx.check_device()  # cleared


# ---------------------------------------------------------------------------
# top-C* and redirect
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,pi,qs,qe,C", [(5000, 64, 4872, 5000, 512), (92160, 256, 91136, 92160, 8192),
                                          (100, 10, 90, 100, 100), (100, 10, 90, 100, 5), (100, 100, 100, 100, 7),
                                          (1, 0, 1, 1, 0), (3000, 0, 3000, 3000, 2999), (777, 5, 700, 777, 200),
                                          (16384, 64, 16000, 16384, 4096), (16385, 64, 16000, 16385, 4096),
                                          (8192, 64, 7680, 8192, 2048), (8193, 64, 7680, 8193, 2048),
                                          (131072, 256, 130048, 131072, 8192), (131073, 256, 130048, 131073, 8192),
                                          (262144, 256, 261120, 262144, 16384), (262145, 256, 261120, 262145, 16384),
                                          (1048576, 256, 1047552, 1048576, 65536)])
def test_topk_exact_on_same_scores(ctx, N, pi, qs, qe, C):
    """The one-CTA, 8-CTA cluster, 16-CTA cluster and re-reading paths on both sides of each
    size limit, bit-exact against the oracle on the same (heavily tied) scores."""
    gen = torch.Generator(device="cuda").manual_seed(N + C)
    s = torch.rand(N, generator=gen, device="cuda")
    s = torch.round(s * 50) / 50  # many exact ties
    keep = torch.empty(N, device="cuda", dtype=torch.uint8)
    idx = torch.empty(N, device="cuda", dtype=torch.int32)
    n = ctx.topk_retain(s, pi, qs, qe, C, keep=keep, keep_idx=idx)
    rk, ridx = oracle.topk_retain(s.cpu().double().numpy(), pi, qs, qe, C)
    assert n == len(ridx)
    np.testing.assert_array_equal(keep.cpu().numpy(), rk)
    np.testing.assert_array_equal(idx[:n].cpu().numpy(), ridx)


def test_topk_special_values(ctx):
    vals = [float("nan"), 0.0, -0.0, 0.5, float("nan"), -1.0, float("inf"), float("-inf"), 1e-45, -1e-45]
    s = torch.tensor(vals * 30, device="cuda")
    for C in (0, 5, 33, 150, 299, 300):
        keep = torch.empty(s.numel(), device="cuda", dtype=torch.uint8)
        idx = torch.empty(s.numel(), device="cuda", dtype=torch.int32)
        n = ctx.topk_retain(s, 2, 290, 300, C, keep=keep, keep_idx=idx)
        rk, ridx = oracle.topk_retain(s.cpu().double().numpy(), 2, 290, 300, C)
        np.testing.assert_array_equal(idx[:n].cpu().numpy(), ridx)
        np.testing.assert_array_equal(keep.cpu().numpy(), rk)


def test_redirect_exact_and_in_place(ctx):
    gen = torch.Generator(device="cuda").manual_seed(5)
    N = 10007
    slot = torch.randperm(N, generator=gen, device="cuda").to(torch.int32)
    keep = (torch.rand(N, generator=gen, device="cuda") < 0.3).to(torch.uint8)
    out = torch.empty_like(slot)
    ctx.redirect_slots(slot, keep, N, out)
    ref = oracle.redirect_slots(slot.cpu().numpy(), keep.cpu().numpy(), N)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    ctx.redirect_slots(slot, keep, N, slot)  # aliasing allowed
    np.testing.assert_array_equal(slot.cpu().numpy(), ref)


# ---------------------------------------------------------------------------
# the whole IntentKV step against the oracle's whole step
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "8b", "long"])
def test_intentkv_step_chain(ctx, name):
    w = synth.TOKEN[name]
    inp = synth.token_inputs(w, "cuda")
    # GPU chain: memory -> rule -> top-C* -> redirect
    M = _gpu_memory(ctx, w, inp["turns"])
    rule = torch.empty(w.N, device="cuda")
    ctx.rule_scores(inp["pool"], M, w.L, w.Hq, w.Hkv, w.N, w.D, w.pi, w.q_s, w.q_e, rule,
                    slot_map=inp["slot_map"], n_slots=w.N)
    keep = torch.empty(w.N, device="cuda", dtype=torch.uint8)
    idx = torch.empty(w.N, device="cuda", dtype=torch.int32)
    n = ctx.topk_retain(rule, w.pi, w.q_s, w.q_e, w.C, keep=keep, keep_idx=idx)
    slot_in = inp["slot_map"] if inp["slot_map"] is not None else torch.arange(w.N, device="cuda", dtype=torch.int32)
    slot_out = torch.empty_like(slot_in)
    ctx.redirect_slots(slot_in, keep, w.dead_slot, slot_out)
    torch.cuda.synchronize()
    assert n == w.n_keep
    # oracle chain, all fp64
    M_ref = _oracle_memory(w, inp["turns"])
    sm = None if inp["slot_map"] is None else inp["slot_map"].cpu().numpy()
    rule_ref = oracle.rule_scores(_host(inp["pool"]).ravel(), M_ref, w.L, w.Hq, w.Hkv, w.N, w.D, w.pi, w.q_s, w.q_e,
                                  slot_map=sm)
    assert_scores_close(f64(rule), rule_ref, what="rule_j chain")
    rk, ridx = oracle.topk_retain(rule_ref, w.pi, w.q_s, w.q_e, w.C)
    forced = _forced(w)
    kept_cand = [j for j in ridx if not forced(j)]
    kth = min(rule_ref[kept_cand]) if kept_cand else 0.0
    assert_keep_sets_match(idx[:n].cpu().numpy(), ridx, rule_ref, kth, forced)
    # redirect consistent with the GPU keep mask, and with the oracle's away from ties
    so = slot_out.cpu().numpy()
    si = slot_in.cpu().numpy()
    km = keep.cpu().numpy().astype(bool)
    assert np.array_equal(so[km], si[km]) and np.all(so[~km] == w.dead_slot)
    assert (so == w.dead_slot).sum() == w.N - n
