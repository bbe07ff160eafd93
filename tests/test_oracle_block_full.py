"""The stored full-size oracle R_b (tests/golden/block_scores_full.npz) and the script that
writes it: the script's multi-process run equals the oracle's own block_scores bit for bit on
small workloads, and the stored vectors keep the invariants the pages fix (KVMEM page, "design
and trade-offs" section: a softmax over the candidate blocks per query row)."""
import os
import sys

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, GOLDEN)
import make_block_scores_full as mk  # noqa: E402


@pytest.mark.parametrize("name,kw", [
    ("ws1m", dict(L=3, Hq=6, Hkv=2, n_blocks=300, M=20, k=64, n_recent=8, new_tokens=64)),
    ("meank262k", dict(L=2, Hq=4, Hkv=2, n_blocks=120, M=12, k=16, n_recent=4)),
])
def test_script_equals_oracle_block_scores(name, kw):
    w = synth.scaled(synth.BLOCK[name], **kw)
    pairs = [(0, 0), (w.L - 1, w.Hkv - 1)]
    out = mk.run(name, 2, w=w, pairs=pairs)
    lay = [synth.portable_block_layer(w, l) for l in range(w.L)]
    q = np.stack([x["q"] for x in lay])
    ix = np.stack([x["index"] for x in lay]) if w.incremental else oracle.meank_build(np.stack([x["raw"] for x in lay]),
                                                                                      w.block)
    R, part = oracle.block_scores(q, ix, w.n_blocks, w.n_sink, w.n_recent, return_partial=True)
    assert np.array_equal(out[name + "_R"], R)
    assert np.array_equal(out[name + "_mass"], part[[l * w.Hkv + g for l, g in pairs]])
    assert str(out[name + "_sha256"]) == synth.portable_digest([synth.portable_layer_digest(x) for x in lay])


@pytest.mark.parametrize("name", ["meank262k", "ws1m"])
def test_stored_values_keep_the_invariants(name):
    g = np.load(os.path.join(GOLDEN, "block_scores_full.npz"))
    w = synth.BLOCK[name]
    R, mass, lg = g[name + "_R"], g[name + "_mass"], g[name + "_mass_lg"]
    G = w.Hq // w.Hkv
    assert R.shape == (w.n_blocks,) and mass.shape == (len(lg), w.n_blocks)
    # each query row's softmax over the candidates sums to 1: sum R_b = M, each mass row = G*M
    assert abs(R.sum() - w.M) < 1e-9 * w.M
    assert np.all(np.abs(mass.sum(axis=1) - G * w.M) < 1e-9 * G * w.M)
    # sink and recent blocks take no part in the softmax
    c0, c1 = w.n_sink, w.n_blocks - w.n_recent
    assert np.all(R[:c0] == 0) and np.all(R[c1:] == 0) and np.all(R[c0:c1] > 0)
    assert np.all(mass[:, :c0] == 0) and np.all(mass[:, c1:] == 0)
    # a mass row is at most G*M per block, and R_b averages all L*Hq heads
    assert np.all(mass <= G * w.M) and R.max() <= w.M
    assert {(0, 0), (w.L - 1, w.Hkv - 1)} <= {tuple(x) for x in lg.tolist()}
    assert len(str(g[name + "_sha256"])) == 64
