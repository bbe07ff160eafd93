"""Parity of the CUDA KVMEM path (Mean-K build, block scores R_b, working-set
selection, re-RoPE scatter) with the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_keep_sets_match, assert_scores_close, bf16_ulp, bits, f64

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


def _bf16_within(got_bits, ref_bits, max_ulp, what, floor=None):
    """|got - ref| <= max_ulp bf16 ulps of ref (ulp taken at max(|ref|, floor))."""
    got, ref = oracle.bf16_to_f64(got_bits), oracle.bf16_to_f64(ref_bits)
    mag = np.abs(ref) if floor is None else np.maximum(np.abs(ref), floor)
    err = np.abs(got - ref)
    bad = np.flatnonzero(err > max_ulp * bf16_ulp(mag) * (1 + 1e-12))
    assert bad.size == 0, f"{what}: {bad.size} of {ref.size} beyond {max_ulp} ulp, first {got.flat[bad[0]]} vs {ref.flat[bad[0]]}"
    return float((got == ref).mean())


# ---------------------------------------------------------------------------
# Mean-K
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,block,first", [(32 * 37 + 5, 32, 0), (64, 32, 3), (1000, 16, 10), (31, 32, 0), (4096, 64, 1)])
def test_meank_parity_small(ctx, T, block, first):
    gen = torch.Generator(device="cuda").manual_seed(T)
    L, Hkv, D = 2, 3, 128
    k = (torch.randn((L, Hkv, T, D), generator=gen, device="cuda") +
         torch.randn((L, Hkv, 1, D), generator=gen, device="cuda")).to(torch.bfloat16)
    nb = (T + block - 1) // block
    Bcap = first + nb + 2
    index = torch.full((L, Hkv, Bcap, D), 3.0, device="cuda", dtype=torch.bfloat16)  # canary outside
    ctx.meank_build(k, block, index, first_block=first)
    ref = oracle.meank_build(bits(k), block, index=bits(index), first_block=first)
    exact = _bf16_within(bits(index), ref, 1, "Mean-K")
    assert exact > 0.999
    got = bits(index)
    assert np.array_equal(got[:, :, :first], ref[:, :, :first]) and np.array_equal(got[:, :, first + nb:], ref[:, :, first + nb:])


@pytest.mark.parametrize("style", [kv.ROPE_NEOX, kv.ROPE_INTERLEAVED])
@pytest.mark.parametrize("D", [64, 128])
def test_meank_de_rope_parity(ctx, style, D):
    gen = torch.Generator(device="cuda").manual_seed(D + style)
    L, Hkv, T = 2, 2, 32 * 9
    k = torch.randn((L, Hkv, T, D), generator=gen, device="cuda").to(torch.bfloat16)
    pos = torch.randint(0, 2 ** 24, (T,), generator=gen, device="cuda", dtype=torch.int32)
    index = torch.zeros((L, Hkv, 9, D), device="cuda", dtype=torch.bfloat16)
    ctx.meank_build(k, 32, index, src_pos=pos, rope_base=1e6, rope_style=style)
    ref = oracle.meank_build(bits(k), 32, Bcap=9, src_pos=pos.cpu().numpy(), rope_base=1e6, rope_style=style)
    _bf16_within(bits(index), ref, 2, "Mean-K de-RoPE", floor=2.0 ** -9)


def test_meank_full_size_sampled(ctx):
    """The 262144-token build at full size; sampled (l, g) slices against the oracle."""
    w = synth.BLOCK["meank262k"]
    inp = synth.block_inputs(w, "cuda")
    index = inp["index"]
    ctx.meank_build(inp["raw"], w.block, index)
    torch.cuda.synchronize()
    for l, g in [(0, 0), (31, 5), (63, 7)]:
        k = bits(inp["raw"][l:l + 1, g:g + 1])
        ref = oracle.meank_build(k, w.block)
        _bf16_within(bits(index[l:l + 1, g:g + 1]), ref, 1, f"Mean-K full l={l} g={g}")


def test_meank_incremental_equals_full(ctx):
    gen = torch.Generator(device="cuda").manual_seed(11)
    L, Hkv, T, D = 2, 2, 32 * 20, 128
    k = torch.randn((L, Hkv, T, D), generator=gen, device="cuda").to(torch.bfloat16)
    full = torch.zeros((L, Hkv, 20, D), device="cuda", dtype=torch.bfloat16)
    ctx.meank_build(k, 32, full)
    inc = torch.zeros_like(full)
    ctx.meank_build(k[:, :, :32 * 12].contiguous(), 32, inc)
    ctx.meank_build(k[:, :, 32 * 12:].contiguous(), 32, inc, first_block=12)
    assert torch.equal(full, inc)


# ---------------------------------------------------------------------------
# block scores R_b
# ---------------------------------------------------------------------------

def _bs_inputs(L, Hq, Hkv, M, Bcap, seed, offset=0.5):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((L, Hq, M, 128), generator=gen, device="cuda").to(torch.bfloat16)
    ix = (torch.randn((L, Hkv, Bcap, 1, 128), generator=gen, device="cuda").squeeze(3) * offset +
          torch.randn((L, Hkv, Bcap, 128), generator=gen, device="cuda") * 0.18).to(torch.bfloat16)
    return q, ix


@pytest.mark.parametrize("L,Hq,Hkv,M,nb,S,Rc", [(2, 10, 2, 40, 300, 4, 10), (1, 8, 8, 130, 257, 0, 0),
                                                 (2, 5, 1, 64, 1000, 4, 64), (1, 4, 2, 1, 5, 1, 1),
                                                 (1, 2, 1, 200, 129, 0, 128), (3, 6, 3, 17, 650, 100, 3)])
def test_block_scores_parity_small(ctx, L, Hq, Hkv, M, nb, S, Rc):
    Bcap = nb + 3
    q, ix = _bs_inputs(L, Hq, Hkv, M, Bcap, seed=nb + M)
    R = torch.empty(nb, device="cuda")
    part = torch.empty((L * Hkv, nb), device="cuda")
    ctx.block_scores(q, ix, nb, S, Rc, R, R_partial=part)
    Rref, pref = oracle.block_scores(bits(q), bits(ix), nb, S, Rc, return_partial=True)
    assert_scores_close(f64(R), Rref, what="R_b")
    assert_scores_close(f64(part), pref, what="R_b partial")
    ncand = max(0, nb - S - Rc)
    if ncand:
        assert abs(f64(R).sum() - M) < 1e-3 * M


def test_block_scores_large_logits(ctx):
    """Queries and index scaled up so logits span tens of units (online max path)."""
    q, ix = _bs_inputs(1, 4, 1, 33, 400, seed=5, offset=3.0)
    q = (q.float() * 3).to(torch.bfloat16)
    R = torch.empty(400, device="cuda")
    ctx.block_scores(q, ix, 400, 2, 2, R)
    assert_scores_close(f64(R), oracle.block_scores(bits(q), bits(ix), 400, 2, 2), what="R_b large logits")


def test_block_scores_row_far_below_its_warp(ctx):
    """Query rows whose logits lie far below the other rows of their 64-row slice:
    one zero row (all logits 0) and one tiny row among rows scaled so that their
    largest logits reach about 140 (log2).  Under the row pass's shared reference
    the zero row's terms flush to zero, so only the exact pass over the marked
    unit gets its total right.  Rows 256..511 form the second unit of each
    (layer, kv head); the first and third units hold no such row and are not redone."""
    L, Hq, Hkv, M, nb = 2, 2, 1, 300, 700
    gen = torch.Generator(device="cuda").manual_seed(77)
    q = torch.randn((L, Hq, M, 128), generator=gen, device="cuda") * 30.0
    ix = torch.randn((L, Hkv, nb, 128), generator=gen, device="cuda")
    q[:, 1, 0] = 0.0                # row 300 of each (l, g): logits exactly 0
    q[:, 1, 5] *= 1e-3              # row 305: logits near 0
    q, ix = q.to(torch.bfloat16), ix.to(torch.bfloat16)
    R = torch.empty(nb, device="cuda")
    part = torch.empty((L * Hkv, nb), device="cuda")
    ctx.block_scores(q, ix, nb, 2, 2, R, R_partial=part)
    ctx.check_device()
    Rref, pref = oracle.block_scores(bits(q), bits(ix), nb, 2, 2, return_partial=True)
    assert_scores_close(f64(part), pref, what="R_b partial, rows far below their slice")
    assert_scores_close(f64(R), Rref, what="R_b, rows far below their slice")


def test_block_scores_every_unit_redone(ctx):
    """A zero query row in every 64-row slice, among rows whose logits reach about 140
    (log2): every row-pass unit of every (layer, kv head) is marked, so the exact pass redoes
    all of them (several units per CTA, none skipped) and must still match the oracle."""
    L, Hq, Hkv, M, nb = 2, 2, 1, 600, 700
    gen = torch.Generator(device="cuda").manual_seed(79)
    q = torch.randn((L, Hq, M, 128), generator=gen, device="cuda") * 30.0
    ix = torch.randn((L, Hkv, nb, 128), generator=gen, device="cuda")
    rows = q.view(L, Hkv, Hq // Hkv * M, 128)
    rows[:, :, ::64] = 0.0          # one zero row per 64-row slice of every unit
    q, ix = q.to(torch.bfloat16), ix.to(torch.bfloat16)
    R = torch.empty(nb, device="cuda")
    part = torch.empty((L * Hkv, nb), device="cuda")
    ctx.block_scores(q, ix, nb, 2, 2, R, R_partial=part)
    ctx.check_device()
    Rref, pref = oracle.block_scores(bits(q), bits(ix), nb, 2, 2, return_partial=True)
    assert_scores_close(f64(part), pref, what="R_b partial, every unit redone")
    assert_scores_close(f64(R), Rref, what="R_b, every unit redone")


@pytest.mark.parametrize("v", [2.6, 3.0])
def test_block_scores_logit_jump_beyond_headroom(ctx, v):
    """A block in the second tile whose logits exceed the first tile's by about 110
    (v = 2.6) or 147 (v = 3.0) in log2 units.  At 110 the row pass's sums grow to about
    2^100 and stay finite; at 147 its terms overflow, the unit is marked, and the exact
    pass (a reference per row with more headroom) gets every total right."""
    L, Hq, Hkv, M, nb = 1, 4, 2, 70, 400
    gen = torch.Generator(device="cuda").manual_seed(78)
    q = torch.full((L, Hq, M, 128), v, device="cuda") + 0.1 * torch.randn((L, Hq, M, 128), generator=gen,
                                                                           device="cuda")
    ix = 0.05 * torch.randn((L, Hkv, nb, 128), generator=gen, device="cuda")
    ix[:, :, 2 + 200] = v           # candidate 200: second tile of 128
    q, ix = q.to(torch.bfloat16), ix.to(torch.bfloat16)
    R = torch.empty(nb, device="cuda")
    ctx.block_scores(q, ix, nb, 2, 2, R)
    ctx.check_device()
    Rref = oracle.block_scores(bits(q), bits(ix), nb, 2, 2)
    assert Rref[202] > 0.99 * Rref.sum()
    assert_scores_close(f64(R), Rref, what="R_b, logit jump")


@pytest.mark.parametrize("name", ["meank262k", "ws1m"])
def test_block_scores_full_size_sampled(ctx, name):
    """Full-size R_b: invariants at full size, and sampled (l, g) masses against the oracle."""
    w = synth.BLOCK[name]
    inp = synth.block_inputs(w, "cuda", with_staging=False)
    index = inp["index"]
    if w.incremental:
        ctx.meank_build(inp["raw"], w.block, index, first_block=w.first_new_block)
    else:
        ctx.meank_build(inp["raw"], w.block, index)
    R = torch.empty(w.n_blocks, device="cuda")
    part = torch.empty((w.L * w.Hkv, w.n_blocks), device="cuda")
    ctx.block_scores(inp["q"], index, w.n_blocks, w.n_sink, w.n_recent, R, R_partial=part)
    torch.cuda.synchronize()
    Rh = f64(R)
    assert abs(Rh.sum() - w.M) < 1e-3 * w.M
    assert np.all(Rh[:w.n_sink] == 0) and np.all(Rh[w.n_blocks - w.n_recent:] == 0) and np.all(Rh >= 0)
    ph = f64(part)
    np.testing.assert_allclose(ph.sum(axis=0) / (w.L * w.Hq), Rh, rtol=1e-4, atol=1e-9)
    samples = [(0, 0), (w.L - 1, w.Hkv - 1)] if name == "meank262k" else [(w.L // 2, 3)]
    for l, g in samples:
        q_lg = bits(inp["q"][l:l + 1])
        ix_lg = bits(index[l:l + 1])
        ref = oracle.block_mass(q_lg, ix_lg, w.n_blocks, w.n_sink, w.n_recent, 0, g)
        assert_scores_close(ph[l * w.Hkv + g], ref, what=f"mass l={l} g={g}")


# ---------------------------------------------------------------------------
# selection
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("nb,S,Rc,k", [(8192, 4, 64, 1024), (32768, 4, 128, 2048), (100, 4, 10, 200), (50, 30, 30, 5),
                                       (1, 0, 0, 1), (1000, 0, 0, 0), (777, 3, 5, 769),
                                       (16384, 4, 64, 1024), (16385, 4, 64, 1024)])
def test_select_exact_on_same_scores(ctx, nb, S, Rc, k):
    gen = torch.Generator(device="cuda").manual_seed(nb + k)
    R = torch.round(torch.rand(nb, generator=gen, device="cuda") * 100) / 100
    ids = torch.empty(nb, device="cuda", dtype=torch.int32)
    n = ctx.select_blocks(R, S, Rc, k, ids)
    ref = oracle.select_blocks(R.cpu().double().numpy(), S, Rc, k)
    assert n == len(ref)
    np.testing.assert_array_equal(ids[:n].cpu().numpy(), ref)


# ---------------------------------------------------------------------------
# re-RoPE scatter
# ---------------------------------------------------------------------------

def _scatter_check(ctx, k_src, src_block, dst_page, dst_pos0, P, page, base, style, n_check=None):
    L, Hkv, T, D = k_src.shape
    pool = torch.randn((L, P, page, Hkv, D), device="cuda").to(torch.bfloat16)  # canary contents
    before = bits(pool)
    ctx.rerope_scatter(k_src, src_block, dst_page, dst_pos0, pool, base, style)
    ctx.check_device()
    got = bits(pool)
    sb, dp, d0 = src_block.cpu().numpy(), dst_page.cpu().numpy(), dst_pos0.cpu().numpy()
    untouched = np.setdiff1d(np.arange(P), dp)
    assert np.array_equal(got[:, untouched], before[:, untouched])
    # sampled entries: evenly spread, with the first and the last (the largest compact positions)
    sel = np.arange(len(sb)) if n_check is None else np.unique(np.linspace(0, len(sb) - 1, n_check).astype(int))
    ks = bits(k_src)
    for i in sel:
        ref = oracle.rerope_scatter(ks, sb[i:i + 1], np.array([0], np.int32), d0[i:i + 1],
                                    np.zeros((L, 1, page, Hkv, D), np.uint16), page, base, style)
        _bf16_within(got[:, dp[i]], ref[:, 0], 2, f"re-RoPE entry {i}")


@pytest.mark.parametrize("style", [kv.ROPE_NEOX, kv.ROPE_INTERLEAVED])
def test_rerope_parity_small(ctx, style):
    gen = torch.Generator(device="cuda").manual_seed(21 + style)
    L, Hkv, D, page, nblk, P = 3, 2, 128, 32, 12, 9
    k = torch.randn((L, Hkv, nblk * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    src_block = torch.tensor([11, 0, 5, 7, 3], device="cuda", dtype=torch.int32)
    dst_page = torch.tensor([8, 1, 0, 4, 6], device="cuda", dtype=torch.int32)
    dst_pos0 = torch.tensor([0, 32, 64, 69728, 2 ** 24 - 32], device="cuda", dtype=torch.int32)
    _scatter_check(ctx, k, src_block, dst_page, dst_pos0, P, page, 1e6, style)


@pytest.mark.parametrize("D,page", [(64, 16), (256, 8), (16, 4)])
def test_rerope_shapes(ctx, D, page):
    gen = torch.Generator(device="cuda").manual_seed(D)
    L, Hkv, nblk, P = 2, 3, 6, 5
    k = torch.randn((L, Hkv, nblk * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    src_block = torch.tensor([5, 2, 0], device="cuda", dtype=torch.int32)
    dst_page = torch.tensor([4, 0, 2], device="cuda", dtype=torch.int32)
    dst_pos0 = torch.tensor([7, 1000, 123456], device="cuda", dtype=torch.int32)
    _scatter_check(ctx, k, src_block, dst_page, dst_pos0, P, page, 1e4, kv.ROPE_NEOX)


def test_rerope_bad_entries_flagged_and_skipped(ctx):
    L, Hkv, D, page = 1, 1, 64, 8
    k = torch.ones((L, Hkv, 4 * page, D), device="cuda", dtype=torch.bfloat16)
    pool = torch.zeros((L, 3, page, Hkv, D), device="cuda", dtype=torch.bfloat16)
    ctx.rerope_scatter(k, torch.tensor([4], device="cuda", dtype=torch.int32),
                       torch.tensor([0], device="cuda", dtype=torch.int32),
                       torch.tensor([0], device="cuda", dtype=torch.int32), pool, 1e4)
    with pytest.raises(kv.KvselError):
        ctx.check_device()
    assert torch.all(pool == 0)
    ctx.rerope_scatter(k, torch.tensor([0], device="cuda", dtype=torch.int32),
                       torch.tensor([3], device="cuda", dtype=torch.int32),
                       torch.tensor([0], device="cuda", dtype=torch.int32), pool, 1e4)
    with pytest.raises(kv.KvselError):
        ctx.check_device()


def test_rerope_full_size_incremental_sampled(ctx):
    """The 1M-workspace scatter at full size: 2048 staged blocks into a shuffled pool."""
    w = synth.BLOCK["ws1m"]
    inp = synth.block_inputs(w, "cuda")
    sb, dp, d0 = synth.scatter_plan_incremental(w, inp["page_perm"])
    _scatter_check(ctx, inp["staging"], sb, dp, d0, inp["pool"].shape[1], w.block, w.rope_base, kv.ROPE_NEOX,
                   n_check=64)


# ---------------------------------------------------------------------------
# the whole KVMEM step against the oracle's whole step (reduced sizes)
# ---------------------------------------------------------------------------

def test_kvmem_step_chain(ctx):
    w = synth.scaled(synth.BLOCK["meank262k"], L=2, Hq=10, Hkv=2, n_blocks=300, M=48, k=50, n_recent=8,
                     new_tokens=300 * 32)
    inp = synth.block_inputs(w, "cuda")
    index = inp["index"]
    ctx.meank_build(inp["raw"], w.block, index)
    R = torch.empty(w.n_blocks, device="cuda")
    ctx.block_scores(inp["q"], index, w.n_blocks, w.n_sink, w.n_recent, R)
    ids = torch.empty(w.n_sel, device="cuda", dtype=torch.int32)
    n = ctx.select_blocks(R, w.n_sink, w.n_recent, w.k, ids)
    dst_page, dst_pos0 = synth.scatter_plan_full(w, inp["page_perm"])
    pool = inp["pool"]
    ctx.rerope_scatter(inp["raw"], ids, dst_page, dst_pos0, pool, w.rope_base)
    torch.cuda.synchronize()
    assert n == w.n_sel
    # oracle chain
    ix_ref = oracle.meank_build(bits(inp["raw"]), w.block)
    R_ref = oracle.block_scores(bits(inp["q"]), ix_ref, w.n_blocks, w.n_sink, w.n_recent)
    assert_scores_close(f64(R), R_ref, what="R_b chain")
    ids_ref = oracle.select_blocks(R_ref, w.n_sink, w.n_recent, w.k)
    cand = [b for b in ids_ref if w.n_sink <= b < w.n_blocks - w.n_recent]
    kth = min(R_ref[cand])
    forced = lambda b: b < w.n_sink or b >= w.n_blocks - w.n_recent  # noqa: E731
    assert_keep_sets_match(ids.cpu().numpy(), ids_ref, R_ref, kth, forced, what="working set")
    # scatter of the GPU's own working set, checked entry by entry
    got = bits(pool)
    ids_np = ids.cpu().numpy()
    ks = bits(inp["raw"])
    for r in range(0, n, 7):
        ref = oracle.rerope_scatter(ks, ids_np[r:r + 1], np.array([0], np.int32), np.array([r * w.block], np.int32),
                                    np.zeros((w.L, 1, w.block, w.Hkv, w.D), np.uint16), w.block, w.rope_base)
        _bf16_within(got[:, dst_page[r].item()], ref[:, 0], 2, f"scatter rank {r}")
