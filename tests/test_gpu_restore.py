"""Parity of the CUDA KVMEM restore path (differential working-set update,
incoming-block restore with V, in-place position shift) with the fp64 oracle,
through the C ABI."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import bf16_ulp, bits

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KEYS = ("in_rank", "in_page", "mv_rank", "mv_shift")


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = kv.Context(0)
    yield c
    c.close()


def _i32(a):
    return torch.as_tensor(np.asarray(a, np.int32), device="cuda")


def _diff_pair(ctx, prev, pages, new, P, page):
    out = ctx.workset_diff(_i32(prev), _i32(pages), _i32(new), P, page)
    ctx.check_device()
    ref = oracle.workset_diff(prev, pages, new, P, page)
    counts = out["counts"].cpu().numpy()
    n_in, n_mv, n_out = (int(c) for c in counts)
    assert (n_in, n_mv, n_out) == (ref["in_rank"].size, ref["mv_rank"].size, ref["out_page"].size)
    n_new = len(new)
    assert out["new_pages"].cpu().numpy()[:n_new].tolist() == ref["new_pages"].tolist()
    assert out["shift"].cpu().numpy()[:n_new].tolist() == ref["shift"].tolist()
    for key, n in zip(KEYS, (n_in, n_in, n_mv, n_mv)):
        assert out[key].cpu().numpy()[:n].tolist() == ref[key].tolist(), key
    assert out["out_page"].cpu().numpy()[:n_out].tolist() == ref["out_page"].tolist()
    return out, ref


def _bf16_within(got_bits, ref_bits, max_ulp, what, floor=None):
    got, ref = oracle.bf16_to_f64(got_bits), oracle.bf16_to_f64(ref_bits)
    mag = np.abs(ref) if floor is None else np.maximum(np.abs(ref), floor)
    err = np.abs(got - ref)
    bad = np.flatnonzero(err > max_ulp * bf16_ulp(mag) * (1 + 1e-12))
    assert bad.size == 0, f"{what}: {bad.size} of {ref.size} beyond {max_ulp} ulp, first {got.flat[bad[0]]} vs {ref.flat[bad[0]]}"


def _pair_mag(raw_rows, style=kv.ROPE_NEOX):
    """Norm of each component's rotation pair (rotation keeps it), per component."""
    x = oracle.bf16_to_f64(raw_rows)
    D = x.shape[-1]
    if style == kv.ROPE_NEOX:
        n = np.sqrt(x[..., :D // 2] ** 2 + x[..., D // 2:] ** 2)
        return np.concatenate([n, n], axis=-1)
    n = np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2)
    return np.repeat(n, 2, axis=-1)


# --------------------------------------------------------------------------
# differential working-set update: bit-exact
# --------------------------------------------------------------------------

def test_workset_diff_golden(ctx):
    g = json.load(open(os.path.join(GOLDEN, "workset_diff_small.json")))
    _diff_pair(ctx, g["prev_ids"], g["prev_pages"], g["new_ids"], g["P"], g["page"])


@pytest.mark.parametrize("seed,universe,n_prev,n_new,extra", [
    (0, 50, 10, 12, 3), (1, 5000, 2180, 2180, 0), (2, 40000, 2180, 2180, 64), (3, 3000, 0, 1500, 0),
    (4, 3000, 1500, 0, 0), (5, 100000, 3000, 2500, 300000), (6, 4000, 2400, 2400, 1)])
def test_workset_diff_parity(ctx, seed, universe, n_prev, n_new, extra):
    rng = np.random.default_rng(seed)
    prev = np.sort(rng.choice(universe, n_prev, replace=False)).astype(np.int32)
    # the new set keeps about two thirds of the previous one
    keep = prev[rng.random(n_prev) < 0.67]
    fresh = np.setdiff1d(np.arange(universe), prev)
    n_fresh = max(0, n_new - keep.size)
    new = np.sort(np.concatenate([keep[:n_new], rng.choice(fresh, n_fresh, replace=False)])).astype(np.int32)
    P = max(n_prev, new.size) + extra
    pages = rng.choice(P, n_prev, replace=False).astype(np.int32)
    _diff_pair(ctx, prev, pages, new, P, 32)


def test_workset_diff_identical_and_disjoint(ctx):
    ids = np.arange(0, 4000, 3, dtype=np.int32)
    pages = np.random.default_rng(9).permutation(ids.size).astype(np.int32)
    out, _ = _diff_pair(ctx, ids, pages, ids, ids.size, 32)
    assert out["counts"].cpu().tolist() == [0, 0, 0]
    out, _ = _diff_pair(ctx, ids, pages, ids + 1, ids.size, 32)
    assert out["counts"].cpu().tolist() == [ids.size, 0, ids.size]


def test_workset_diff_errors(ctx):
    # more blocks than pages: rejected on the host before any launch
    with pytest.raises(kv.KvselError):
        ctx.workset_diff(_i32([1, 4]), _i32([0, 1]), _i32([0, 1, 4]), 2, 32)
    with pytest.raises(kv.KvselError):
        ctx.workset_diff(_i32([1, 4, 5]), _i32([0, 1, 2]), _i32([1]), 2, 32)
    ctx.check_device()
    # a set that is not ascending, a page held twice, a page outside the pool: device checks
    ctx.workset_diff(_i32([1, 4]), _i32([0, 1]), _i32([4, 1]), 4, 32)
    with pytest.raises(kv.KvselError, match="ascending"):
        ctx.check_device()
    ctx.workset_diff(_i32([1, 4]), _i32([2, 2]), _i32([1, 4]), 4, 32)
    with pytest.raises(kv.KvselError, match="held twice"):
        ctx.check_device()
    ctx.workset_diff(_i32([1, 4]), _i32([0, 9]), _i32([1, 4]), 4, 32)
    with pytest.raises(kv.KvselError, match="page out of range"):
        ctx.check_device()
    ctx.check_device()


# --------------------------------------------------------------------------
# incoming-block restore: K re-rotated (2 bf16 ulp), V bit-exact
# --------------------------------------------------------------------------

@pytest.mark.parametrize("style", [kv.ROPE_NEOX, kv.ROPE_INTERLEAVED])
def test_restore_blocks_parity(ctx, style):
    gen = torch.Generator(device="cuda").manual_seed(31 + style)
    L, Hkv, D, page, nblk, P = 3, 2, 128, 32, 10, 12
    k = torch.randn((L, Hkv, nblk * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn((L, Hkv, nblk * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    kp = torch.randn((L, P, page, Hkv, D), generator=gen, device="cuda").to(torch.bfloat16)
    vp = torch.randn((L, P, page, Hkv, D), generator=gen, device="cuda").to(torch.bfloat16)
    src = np.array([9, 0, 4, 2, 7], np.int32)
    dpg = np.array([11, 3, 0, 6, 5], np.int32)
    pos0 = np.array([0, 32, 69728, 2 ** 24 - 32, 640], np.int32)
    kb, vb = bits(kp), bits(vp)
    ctx.restore_blocks(k, v, _i32(src), _i32(dpg), _i32(pos0), kp, vp, 1e6, style)
    ctx.check_device()
    ref_k, ref_v = oracle.restore_blocks(bits(k), bits(v), src, dpg, pos0, kb, vb, page, 1e6, style)
    assert np.array_equal(bits(vp), ref_v)
    got = bits(kp)
    untouched = np.setdiff1d(np.arange(P), dpg)
    assert np.array_equal(got[:, untouched], kb[:, untouched])
    for i in range(src.size):
        _bf16_within(got[:, dpg[i]], ref_k[:, dpg[i]], 2, f"restore entry {i}")


def test_restore_and_shift_full_size_sampled(ctx):
    """The 1M-workspace restore at full size: 2048 blocks (L64 Hkv8 D128, 32-token pages) restored
    into a shuffled pool of 2180 pages; V compared whole on the device, K on sampled (layer, entry)
    pairs against the oracle; then those pages shifted in place and sampled again."""
    L, Hkv, D, page, nblk, P = 64, 8, 128, 32, 2048, 2180
    gen = torch.Generator(device="cuda").manual_seed(2048)
    k = torch.randn((L, Hkv, nblk * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn((L, Hkv, nblk * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    kp = torch.zeros((L, P, page, Hkv, D), device="cuda", dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    rng = np.random.default_rng(9)
    src = rng.permutation(nblk).astype(np.int32)
    dpg = rng.choice(P, nblk, replace=False).astype(np.int32)
    pos0 = (np.arange(nblk, dtype=np.int32) + 4) * page
    ctx.restore_blocks(k, v, _i32(src), _i32(dpg), _i32(pos0), kp, vp, 1e6)
    ctx.check_device()
    # V: every restored page is the source block's rows, bit for bit
    v_rows = v.view(L, Hkv, nblk, page, D)[:, :, torch.as_tensor(src, device="cuda")].permute(0, 2, 3, 1, 4)
    assert torch.equal(vp[:, torch.as_tensor(dpg, device="cuda")], v_rows)
    del v_rows
    # K: sampled (layer, entry) pairs against the oracle (2 bf16 ulp of the rotation pair norm)
    for l, i in [(0, 0), (17, 1000), (L - 1, nblk - 1)]:
        k_l = bits(k[l:l + 1])
        one = np.zeros((1, 1, page, Hkv, D), np.uint16)
        ref_k, _ = oracle.restore_blocks(k_l, k_l, src[i:i + 1], np.zeros(1, np.int32), pos0[i:i + 1], one, one.copy(),
                                         page, 1e6)
        _bf16_within(bits(kp[l:l + 1, int(dpg[i])]), ref_k[:, 0], 2, f"restored K l={l} entry {i}")
    # in-place shift of every restored page by its own offset
    shifts = rng.integers(-2 ** 16, 2 ** 16, nblk).astype(np.int32)
    samples = [(3, 5), (40, 2047)]
    before = {(l, i): bits(kp[l:l + 1, int(dpg[i])]) for l, i in samples}
    ctx.rerope_shift(kp, _i32(dpg), _i32(shifts), 1e6)
    ctx.check_device()
    for (l, i), b0 in before.items():
        ref = oracle.rerope_shift(b0[:, None], np.zeros(1, np.int32), shifts[i:i + 1], page, 1e6)
        _bf16_within(bits(kp[l:l + 1, int(dpg[i])]), ref[:, 0], 2, f"shifted K l={l} entry {i}")


def test_restore_blocks_device_count(ctx):
    """Entries at or past the device-side count leave their pages untouched."""
    L, Hkv, D, page, P = 2, 2, 64, 16, 6
    gen = torch.Generator(device="cuda").manual_seed(5)
    k = torch.randn((L, Hkv, 4 * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn((L, Hkv, 4 * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    kp = torch.zeros((L, P, page, Hkv, D), device="cuda", dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    n_dev = _i32([2])
    ctx.restore_blocks(k, v, _i32([0, 1, 2, 3]), _i32([5, 4, 3, 2]), _i32([0, 16, 32, 48]), kp, vp, 1e4,
                       n_dev=n_dev)
    ctx.check_device()
    assert torch.all(kp[:, [2, 3]] == 0) and torch.all(vp[:, [2, 3]] == 0)
    assert torch.equal(vp[:, 5], v[:, :, :page].permute(0, 2, 1, 3))


# --------------------------------------------------------------------------
# in-place position shift (2 bf16 ulp)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("style", [kv.ROPE_NEOX, kv.ROPE_INTERLEAVED])
@pytest.mark.parametrize("D,page", [(128, 32), (64, 16), (256, 8)])
def test_rerope_shift_parity(ctx, style, D, page):
    gen = torch.Generator(device="cuda").manual_seed(D + style)
    L, Hkv, P = 3, 2, 9
    pool = torch.randn((L, P, page, Hkv, D), generator=gen, device="cuda").to(torch.bfloat16)
    before = bits(pool)
    pages = np.array([8, 0, 3, 5], np.int32)
    shifts = np.array([32, -64, 2 ** 24 - 1, -(2 ** 20 + 7)], np.int32)
    ctx.rerope_shift(pool, _i32(pages), _i32(shifts), 1e6, style)
    ctx.check_device()
    ref = oracle.rerope_shift(before, pages, shifts, page, 1e6, style)
    got = bits(pool)
    untouched = np.setdiff1d(np.arange(P), pages)
    assert np.array_equal(got[:, untouched], before[:, untouched])
    for i, pg in enumerate(pages):
        _bf16_within(got[:, pg], ref[:, pg], 2, f"shift entry {i}")


def test_rerope_shift_zero_and_bad_entries(ctx):
    pool = torch.randn((1, 3, 4, 1, 32), device="cuda").to(torch.bfloat16)
    before = pool.clone()
    ctx.rerope_shift(pool, _i32([0, 2]), _i32([0, 0]), 1e4)
    ctx.check_device()
    assert torch.equal(pool, before)
    ctx.rerope_shift(pool, _i32([3]), _i32([5]), 1e4)  # page outside the pool
    with pytest.raises(kv.KvselError, match="page"):
        ctx.check_device()
    assert torch.equal(pool, before)


# --------------------------------------------------------------------------
# one whole restore step: diff, move the retained blocks, restore the incoming ones
# --------------------------------------------------------------------------

def test_restore_step_chain(ctx):
    """After the step every rank r of the new working set holds RoPE(raw K, r*page + t)
    and its V: restored blocks within 2 bf16 ulp, moved ones (rounded twice) within
    2 bf16 ulp of their rotation pair's norm."""
    rng = np.random.default_rng(3)
    L, Hkv, D, page, universe = 2, 2, 128, 32, 400
    base = 1e6
    gen = torch.Generator(device="cuda").manual_seed(3)
    raw_k = torch.randn((L, Hkv, universe * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    raw_v = torch.randn((L, Hkv, universe * page, D), generator=gen, device="cuda").to(torch.bfloat16)
    prev = np.sort(rng.choice(universe, 120, replace=False)).astype(np.int32)
    new = np.sort(np.concatenate([prev[rng.random(prev.size) < 0.6],
                                  rng.choice(np.setdiff1d(np.arange(universe), prev), 50, replace=False)])).astype(np.int32)
    P = 180
    prev_pages = rng.choice(P, prev.size, replace=False).astype(np.int32)
    kp = torch.zeros((L, P, page, Hkv, D), device="cuda", dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    # the previous step's pool: block prev[r] in page prev_pages[r] at position r*page
    ctx.restore_blocks(raw_k, raw_v, _i32(prev), _i32(prev_pages), _i32(np.arange(prev.size) * page), kp, vp, base)
    d = ctx.workset_diff(_i32(prev), _i32(prev_pages), _i32(new), P, page)
    n_in, n_mv, _ = (int(c) for c in d["counts"].cpu())
    mv_pages = d["new_pages"][d["mv_rank"][:n_mv].long()]
    ctx.rerope_shift(kp, mv_pages, d["mv_shift"][:n_mv], base)
    in_rank = d["in_rank"][:n_in]
    in_blocks = _i32(new)[in_rank.long()]
    ctx.restore_blocks(raw_k, raw_v, in_blocks, d["in_page"][:n_in], in_rank * page, kp, vp, base)
    ctx.check_device()
    got_k, got_v = bits(kp), bits(vp)
    rk, rv = bits(raw_k), bits(raw_v)
    new_pages = d["new_pages"].cpu().numpy()[:new.size]
    incoming = set(in_rank.cpu().tolist())
    for r in range(0, new.size, 5):
        b, pg = int(new[r]), int(new_pages[r])
        src = slice(b * page, (b + 1) * page)
        assert np.array_equal(got_v[:, pg], rv[:, :, src].transpose(0, 2, 1, 3))
        one = np.zeros((L, 1, page, Hkv, D), np.uint16)
        ref = oracle.rerope_scatter(rk, np.array([b], np.int32), np.array([0], np.int32),
                                    np.array([r * page], np.int32), one, page, base)
        raw_rows = rk[:, :, src].transpose(0, 2, 1, 3)
        if r in incoming:
            _bf16_within(got_k[:, pg], ref[:, 0], 2, f"restored rank {r}")
        else:
            # rounded once at the old position and once after the turn: the first rounding of
            # a pair's larger component reaches its smaller one, so the bound is in ulps of
            # the pair's norm
            _bf16_within(got_k[:, pg], ref[:, 0], 2, f"moved rank {r}", floor=_pair_mag(raw_rows))


# --------------------------------------------------------------------------
# packed, pipelined host -> device rematerialisation
# --------------------------------------------------------------------------

def _host_repo(L, Hkv, n_blocks, page, D, seed, pinned):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn((L, Hkv, n_blocks * page, D), generator=g).to(torch.bfloat16)
    v = torch.randn((L, Hkv, n_blocks * page, D), generator=g).to(torch.bfloat16)
    if pinned:
        k, v = k.pin_memory(), v.pin_memory()
    return k, v


@pytest.mark.parametrize("chunk,threads,pinned,mode", [(1, 1, False, kv.STAGE_AUTO), (7, 4, False, kv.STAGE_PACKED),
                                                       (32, 8, True, kv.STAGE_PACKED), (500, 3, True, kv.STAGE_PACKED),
                                                       (16, 2, True, kv.STAGE_DIRECT), (16, 2, True, kv.STAGE_AUTO)])
def test_stage_restore_equals_device_restore(ctx, chunk, threads, pinned, mode):
    """The staged restore from host memory writes exactly what restore_blocks writes from device memory."""
    L, Hkv, D, page, nrepo, P = 3, 2, 128, 32, 90, 80
    hk, hv = _host_repo(L, Hkv, nrepo, page, D, chunk, pinned)
    rng = np.random.default_rng(chunk)
    n = 60
    blocks = rng.choice(nrepo, n, replace=False).astype(np.int32)
    pages = rng.choice(P, n, replace=False).astype(np.int32)
    pos0 = (rng.permutation(n) * page).astype(np.int32)
    kp = torch.randn((L, P, page, Hkv, D), device="cuda").to(torch.bfloat16)
    vp = torch.randn_like(kp)
    kp2, vp2 = kp.clone(), vp.clone()
    ctx.stage_restore(hk, hv, blocks, pages, pos0, kp, vp, 1e6, chunk_blocks=chunk, gather_threads=threads, mode=mode)
    ctx.check_device()
    ctx.restore_blocks(hk.cuda(), hv.cuda(), _i32(blocks), _i32(pages), _i32(pos0), kp2, vp2, 1e6)
    ctx.check_device()
    assert torch.equal(kp, kp2) and torch.equal(vp, vp2)
    # and a sample against the oracle
    ref_k, ref_v = oracle.restore_blocks(bits(hk), bits(hv), blocks[:3], pages[:3], pos0[:3],
                                         np.zeros((L, P, page, Hkv, D), np.uint16),
                                         np.zeros((L, P, page, Hkv, D), np.uint16), page, 1e6)
    got_k, got_v = bits(kp), bits(vp)
    for i in range(3):
        assert np.array_equal(got_v[:, pages[i]], ref_v[:, pages[i]])
        _bf16_within(got_k[:, pages[i]], ref_k[:, pages[i]], 2, f"staged entry {i}")


def test_stage_restore_repeated_calls_and_growth(ctx):
    """Consecutive calls reuse the staging slots (and grow them) without disturbing queued work."""
    L, Hkv, D, page, nrepo, P = 2, 2, 64, 16, 40, 40
    hk, hv = _host_repo(L, Hkv, nrepo, page, D, 99, False)
    kp = torch.zeros((L, P, page, Hkv, D), device="cuda", dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    for step, chunk in enumerate((2, 2, 9, 3)):
        blocks = np.arange(step * 10, step * 10 + 10, dtype=np.int32)
        ctx.stage_restore(hk, hv, blocks, blocks, blocks * page, kp, vp, 1e4, chunk_blocks=chunk, gather_threads=2)
    ctx.check_device()
    # block b went to page b: pool[l][b][t][g] = repository[l][g][b*page + t]
    assert torch.equal(vp, hv.cuda().permute(0, 2, 1, 3).reshape(L, P, page, Hkv, D))


def test_stage_restore_host_checks(ctx):
    L, Hkv, D, page = 1, 1, 64, 8
    hk, hv = _host_repo(L, Hkv, 4, page, D, 1, False)
    kp = torch.zeros((L, 3, page, Hkv, D), device="cuda", dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    for blocks, pages, pos in (([4], [0], [0]), ([0], [3], [0]), ([0], [0], [2 ** 24 - 4])):
        with pytest.raises(kv.KvselError):
            ctx.stage_restore(hk, hv, np.array(blocks, np.int32), np.array(pages, np.int32), np.array(pos, np.int32),
                              kp, vp, 1e4)
    assert torch.all(kp == 0) and torch.all(vp == 0)
    with pytest.raises(kv.KvselError, match="pinned"):  # direct mode on pageable memory is refused on the host
        ctx.stage_restore(hk, hv, np.array([0], np.int32), np.array([0], np.int32), np.array([0], np.int32), kp, vp,
                          1e4, mode=kv.STAGE_DIRECT)
    ctx.check_device()


# --------------------------------------------------------------------------
# SideQuest cursor-span eviction: bit-exact
# --------------------------------------------------------------------------

def test_span_keep_golden(ctx):
    g = json.load(open(os.path.join(GOLDEN, "span_keep_small.json")))
    keep_in = torch.tensor(g["keep_in"], dtype=torch.uint8, device="cuda")
    out = torch.empty_like(keep_in)
    ctx.span_keep(_i32(g["span_start"]), _i32(g["span_end"]), _i32(g["del_ids"]), g["N"], out, keep_in=keep_in)
    with pytest.raises(kv.KvselError, match="cursor id"):  # id 7 is not a cursor
        ctx.check_device()
    assert out.cpu().tolist() == g["keep_out"]


@pytest.mark.parametrize("seed,N,n_cur,n_del", [(0, 92160, 500, 120), (1, 32768, 6000, 5000), (2, 1, 3, 3),
                                               (3, 70001, 40, 0), (4, 4096, 2, 2)])
def test_span_keep_parity(ctx, seed, N, n_cur, n_del):
    rng = np.random.default_rng(seed)
    start = rng.integers(-50, N + 50, n_cur).astype(np.int32)
    end = (start + rng.integers(0, 2000, n_cur)).astype(np.int32)
    dels = rng.choice(n_cur, n_del, replace=False).astype(np.int32)
    keep_in = (rng.random(N) < 0.7).astype(np.uint8)
    ref, bad = oracle.span_keep(start, end, dels, N, keep_in)
    assert bad == 0
    k = torch.as_tensor(keep_in, device="cuda")
    ctx.span_keep(_i32(start), _i32(end), _i32(dels), N, k, keep_in=k)  # in place
    ctx.check_device()
    assert np.array_equal(k.cpu().numpy(), ref)
    ones = torch.empty(N, dtype=torch.uint8, device="cuda")
    ctx.span_keep(_i32(start), _i32(end), _i32(dels), N, ones)
    ctx.check_device()
    assert np.array_equal(ones.cpu().numpy(), oracle.span_keep(start, end, dels, N)[0])


def test_span_keep_then_redirect(ctx):
    """An IntentKV keep mask, cleared of the deleted cursors' spans, drives the dead-slot redirect."""
    N, dead = 10000, 10000
    rng = np.random.default_rng(8)
    keep = (rng.random(N) < 0.5).astype(np.uint8)
    start = np.array([100, 5000, 9990], np.int32)
    end = np.array([300, 5100, 10010], np.int32)
    slots = rng.permutation(N).astype(np.int32)
    k = torch.as_tensor(keep, device="cuda")
    ctx.span_keep(_i32(start), _i32(end), _i32([0, 2]), N, k, keep_in=k)
    out = torch.empty(N, dtype=torch.int32, device="cuda")
    ctx.redirect_slots(_i32(slots), k, dead, out)
    ctx.check_device()
    ref_keep, _ = oracle.span_keep(start, end, np.array([0, 2], np.int32), N, keep)
    assert np.array_equal(out.cpu().numpy(), oracle.redirect_slots(slots, ref_keep, dead))
