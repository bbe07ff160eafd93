"""Pins of the fp64 oracle's KVMEM half (RoPE, Mean-K index, block scores R_b,
sink/recent/top selection, re-RoPE scatter) against what the page and the
mathematics fix.  CPU only."""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle


def _bf16(x):
    return oracle.bf16_round(np.asarray(x, np.float64))


def _bf16_fast(rng, shape, scale=1.0, offset=None):
    """Random bf16 bits via torch's float32 -> bf16 conversion (library, RNE)."""
    x = rng.standard_normal(shape).astype(np.float32) * scale
    if offset is not None:
        x = x + offset
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# bf16 rounding and RoPE
# --------------------------------------------------------------------------

def test_bf16_round_matches_library_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(2000).astype(np.float32),
                        (rng.standard_normal(500) * 1e-39).astype(np.float32),  # subnormals
                        np.array([0.0, -0.0, 1.0, 65504.0, 3.3e38], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_round(x.astype(np.float64)), ref)


def test_bf16_round_ties_and_single_rounding():
    vals = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -30, -(1.0 + 2 ** -8 + 2 ** -30)]
    assert oracle.bf16_round(vals).tolist() == [0x3F80, 0x3F82, 0x3F81, 0xBF81]


def test_rope_golden(golden):
    g = golden("rope_d4.json")
    for c in g["cases"]:
        style = oracle.ROPE_NEOX if c["style"] == "neox" else oracle.ROPE_INTERLEAVED
        y = oracle.rope_rotate(c["x"], c["pos"], g["base"], style)
        np.testing.assert_allclose(y, c["y"], atol=1e-15)


def _rope_complex(x, pos, base, style):
    """Textbook form: each pair is a complex number multiplied by e^{i pos theta_i}."""
    D = x.shape[-1]
    theta = base ** (-2.0 * np.arange(D // 2) / D)
    if style == oracle.ROPE_NEOX:
        z = x[: D // 2] + 1j * x[D // 2:]
    else:
        z = x[0::2] + 1j * x[1::2]
    z = z * np.exp(1j * pos * theta)
    out = np.empty(D)
    if style == oracle.ROPE_NEOX:
        out[: D // 2], out[D // 2:] = z.real, z.imag
    else:
        out[0::2], out[1::2] = z.real, z.imag
    return out


@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_INTERLEAVED])
def test_rope_properties(style):
    rng = np.random.default_rng(1)
    D = 64
    for pos in [0, 1, 17, 4096, 69759, 999_983]:
        x = rng.standard_normal(D)
        y = oracle.rope_rotate(x, pos, 1e6, style)
        np.testing.assert_allclose(y, _rope_complex(x, pos, 1e6, style), atol=1e-9)
        back = oracle.rope_rotate(y, pos, 1e6, style, inverse=True)
        np.testing.assert_allclose(back, x, atol=1e-12)      # round trip
        if pos == 0:
            np.testing.assert_array_equal(y, x)               # identity
        np.testing.assert_allclose(np.linalg.norm(y), np.linalg.norm(x), rtol=1e-13)
    x = rng.standard_normal(D)
    two = oracle.rope_rotate(oracle.rope_rotate(x, 300, 1e4, style), 700, 1e4, style)
    np.testing.assert_allclose(two, oracle.rope_rotate(x, 1000, 1e4, style), atol=1e-11)


# --------------------------------------------------------------------------
# Mean-K (KVMEM retrieval index)
# --------------------------------------------------------------------------

def test_meank_golden(golden):
    g = golden("meank_tiny.json")
    rows = np.array(g["rows"], np.float64)
    k = _bf16(rows)[None, None]                   # [1,1,T,D]
    index, mean = oracle.meank_build(k, g["block"], return_mean=True)
    np.testing.assert_array_equal(mean[0, 0], g["mean"])
    np.testing.assert_array_equal(oracle.bf16_to_f64(index[0, 0]), g["index_bf16_value"])


def test_meank_equal_rows_linearity_numpy_mean():
    rng = np.random.default_rng(2)
    L, Hkv, T, D, blk = 2, 3, 96, 16, 32
    row = _bf16(rng.standard_normal(D))
    same = np.broadcast_to(row, (L, Hkv, T, D)).copy()
    assert np.array_equal(oracle.meank_build(same, blk), np.broadcast_to(row, (L, Hkv, T // blk, D)))
    X = _bf16_fast(rng, (L, Hkv, T, D))
    Y = _bf16_fast(rng, (L, Hkv, T, D))
    _, mx = oracle.meank_build(X, blk, return_mean=True)
    _, my = oracle.meank_build(Y, blk, return_mean=True)
    ref = oracle.bf16_to_f64(X).reshape(L, Hkv, T // blk, blk, D).mean(axis=3)
    np.testing.assert_allclose(mx, ref, rtol=1e-14, atol=1e-16)
    # linearity of the mean: exact scaling by 2 of bf16 values stays bf16-exact
    _, m2 = oracle.meank_build(_bf16(2.0 * oracle.bf16_to_f64(X) + 0.0), blk, return_mean=True)
    np.testing.assert_allclose(m2, 2.0 * mx, rtol=1e-15)
    # additivity: the mean of X plus the mean of Y equals the mean of the fp64 row sums
    S = oracle.bf16_to_f64(X) + oracle.bf16_to_f64(Y)
    mean_sum = S.reshape(L, Hkv, T // blk, blk, D).mean(axis=3)
    np.testing.assert_allclose(mx + my, mean_sum, rtol=1e-12, atol=1e-15)


def test_meank_incremental_equals_full_and_short_tail():
    rng = np.random.default_rng(3)
    L, Hkv, T, D, blk = 1, 2, 160, 8, 32
    X = _bf16_fast(rng, (L, Hkv, T, D))
    full = oracle.meank_build(X, blk, Bcap=8)
    tail = oracle.meank_build(np.ascontiguousarray(X[:, :, 96:]), blk, index=np.zeros_like(full),
                              first_block=3)
    np.testing.assert_array_equal(tail[:, :, 3:5], full[:, :, 3:5])
    assert np.all(tail[:, :, :3] == 0) and np.all(tail[:, :, 5:] == 0)
    short = oracle.meank_build(np.ascontiguousarray(X[:, :, :70]), blk, Bcap=3, return_mean=True)[1]
    ref = oracle.bf16_to_f64(X[:, :, 64:70]).mean(axis=2)
    np.testing.assert_allclose(short[:, :, 2], ref, rtol=1e-14)


@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_INTERLEAVED])
def test_meank_de_rope(style):
    """With positions, rows are de-rotated (complex form) before averaging."""
    rng = np.random.default_rng(4)
    L, Hkv, T, D, blk = 1, 1, 64, 16, 32
    X = _bf16_fast(rng, (L, Hkv, T, D))
    pos = rng.integers(0, 1_000_000, T).astype(np.int32)
    _, mean = oracle.meank_build(X, blk, src_pos=pos, rope_base=1e6, rope_style=style, return_mean=True)
    rows = oracle.bf16_to_f64(X[0, 0])
    der = np.stack([_rope_complex(rows[t], -float(pos[t]), 1e6, style) for t in range(T)])
    np.testing.assert_allclose(mean[0, 0], der.reshape(2, blk, D).mean(axis=1), atol=1e-9)


# --------------------------------------------------------------------------
# R_b block scores (KVMEM retrieval)
# --------------------------------------------------------------------------

def test_block_scores_golden(golden):
    g = golden("block_scores_tiny.json")
    q = _bf16(g["q"]).reshape(1, 1, 1, g["D"])
    ix = _bf16(g["index"]).reshape(1, 1, g["n_blocks"], g["D"])
    R = oracle.block_scores(q, ix, g["n_blocks"], g["n_sink"], g["n_recent"])
    np.testing.assert_allclose(R, g["R"], rtol=1e-14, atol=1e-16)


def test_block_scores_sum_constant_and_brute_force():
    rng = np.random.default_rng(5)
    L, Hq, Hkv, M, D, nb, Bcap = 2, 6, 2, 5, 16, 40, 48
    q = _bf16_fast(rng, (L, Hq, M, D))
    ix = _bf16_fast(rng, (L, Hkv, Bcap, D), scale=0.5)
    S, Rc = 3, 4
    R, part = oracle.block_scores(q, ix, nb, S, Rc, return_partial=True)
    assert abs(R.sum() - M) < 1e-12                               # sum over C of R_b = M
    assert np.all(R[:S] == 0) and np.all(R[nb - Rc:] == 0)
    np.testing.assert_allclose(part.sum(axis=0) / (L * Hq), R, rtol=1e-13)
    # brute force with the library softmax
    G = Hq // Hkv
    qf, kf = oracle.bf16_to_f64(q), oracle.bf16_to_f64(ix)
    ref = np.zeros(nb)
    for l in range(L):
        for h in range(Hq):
            logits = qf[l, h] @ kf[l, h // G, S:nb - Rc].T / np.sqrt(D)   # [M, |C|]
            ref[S:nb - Rc] += softmax(logits, axis=1).sum(axis=0)
    np.testing.assert_allclose(R, ref / (L * Hq), rtol=1e-12, atol=1e-16)
    # constant index -> every candidate gets M/|C|
    const = np.broadcast_to(ix[:, :, :1], ix.shape).copy()
    Rc_ = oracle.block_scores(q, const, nb, S, Rc)
    np.testing.assert_allclose(Rc_[S:nb - Rc], M / (nb - S - Rc), rtol=1e-13)


def test_block_scores_single_head_is_softmax_and_gqa():
    rng = np.random.default_rng(6)
    D, nb = 8, 12
    q = _bf16_fast(rng, (1, 1, 1, D))
    ix = _bf16_fast(rng, (1, 1, nb, D))
    R = oracle.block_scores(q, ix, nb, 0, 0)
    logits = oracle.bf16_to_f64(ix[0, 0]) @ oracle.bf16_to_f64(q[0, 0, 0]) / np.sqrt(D)
    np.testing.assert_allclose(R, softmax(logits), rtol=1e-13)
    # GQA: heads 0,1 -> kv 0, heads 2,3 -> kv 1
    q = np.zeros((1, 4, 1, 4)); q[0, :2, 0, 0] = 1; q[0, 2:, 0, 1] = 1
    ix = np.zeros((1, 2, 6, 4)); ix[0, 0, 2, 0] = 60; ix[0, 1, 4, 1] = 60
    R = oracle.block_scores(_bf16(q), _bf16(ix), 6, 0, 0)
    assert R[2] > 0.499 and R[4] > 0.499


def test_block_scores_empty_candidates():
    rng = np.random.default_rng(7)
    q = _bf16_fast(rng, (1, 2, 3, 8))
    ix = _bf16_fast(rng, (1, 1, 10, 8))
    assert np.all(oracle.block_scores(q, ix, 10, 6, 4) == 0)


# --------------------------------------------------------------------------
# block selection
# --------------------------------------------------------------------------

def test_select_golden(golden):
    g = golden("select_blocks_tiny.json")
    ids = oracle.select_blocks(np.array(g["R"]), g["n_sink"], g["n_recent"], g["k"])
    assert ids.tolist() == g["ids"]


@pytest.mark.parametrize("seed", range(5))
def test_select_invariants(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(1, 400))
    S = int(rng.integers(0, 10)); Rc = int(rng.integers(0, 20)); k = int(rng.integers(0, 100))
    R = np.round(rng.random(nb), 2)
    ids = oracle.select_blocks(R, S, Rc, k)
    forced = set(range(min(S, nb))) | set(range(max(nb - Rc, 0), nb))
    cand = [b for b in range(nb) if b not in forced]
    assert forced <= set(ids.tolist()) and np.all(np.diff(ids) > 0)
    assert len(ids) == len(forced) + min(k, len(cand))
    ref = sorted(cand, key=lambda b: (-R[b], b))[:k]
    assert sorted(set(ids.tolist()) - forced) == sorted(ref)


# --------------------------------------------------------------------------
# re-RoPE scatter (KVMEM position-consistent rebuild)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("style", [oracle.ROPE_NEOX, oracle.ROPE_INTERLEAVED])
def test_rerope_scatter_mapping_and_untouched(style):
    rng = np.random.default_rng(8)
    L, Hkv, T, D, page, P = 2, 3, 8 * 4, 16, 4, 10
    src = _bf16_fast(rng, (L, Hkv, T, D))
    pool = _bf16_fast(rng, (L, P, page, Hkv, D))
    src_block = np.array([5, 1, 7], np.int32)
    dst_page = np.array([9, 0, 4], np.int32)
    dst_pos0 = np.array([0, 4, 800], np.int32)
    out = oracle.rerope_scatter(src, src_block, dst_page, dst_pos0, pool, page, 1e6, style)
    untouched = [p for p in range(P) if p not in dst_page]
    np.testing.assert_array_equal(out[:, untouched], pool[:, untouched])
    sf = oracle.bf16_to_f64(src)
    for i in range(3):
        for l in range(L):
            for t in range(page):
                for g in range(Hkv):
                    row = sf[l, g, src_block[i] * page + t]
                    ref = _rope_complex(row, dst_pos0[i] + t, 1e6, style)
                    got = oracle.bf16_to_f64(out[l, dst_page[i], t, g])
                    # one rounding to bf16 of the exact rotation: within half an ulp
                    ulp = np.spacing(np.maximum(np.abs(ref), 1e-30).astype(np.float32)) * 2 ** 16
                    assert np.all(np.abs(got - ref) <= 0.5 * ulp + 1e-12)
    # position 0 keeps the raw rows bit for bit
    out0 = oracle.rerope_scatter(src, np.array([2], np.int32), np.array([3], np.int32),
                                 np.array([0], np.int32), pool, page, 1e6, style)
    assert np.array_equal(out0[:, 3, 0], src[:, :, 2 * page])
