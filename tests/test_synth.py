"""The seeded input recipe: workload sizes and derived counts as the workload table states them,
and generators that are deterministic, shaped as documented and structured as described
(paged slot maps, outlier channels, block offsets, incremental index, scatter plans)."""
import dataclasses

import torch

import synth


def test_token_workload_counts():
    t, e, lg = synth.TOKEN["tiny"], synth.TOKEN["8b"], synth.TOKEN["long"]
    # forced set F = [0, pi) U [q_s, q_e), candidates H, C* = max(0, C - |F|)
    assert (t.n_forced, t.n_cand, t.C - t.n_forced) == (192, 1856, 320)
    assert (e.n_forced, e.n_cand, e.C - e.n_forced) == (768, 32000, 7424)
    assert (lg.n_forced, lg.n_cand, lg.C - lg.n_forced) == (1280, 90880, 6912)
    assert t.dead_slot == 2048 and e.dead_slot == 32768
    assert e.k_bytes() == 36 * 32768 * 8 * 128 * 2 and lg.k_bytes() == 48 * 92160 * 8 * 128 * 2
    assert e.n_keep == 768 + 7424


def test_block_workload_counts():
    m, w = synth.BLOCK["meank262k"], synth.BLOCK["ws1m"]
    assert (m.n_cand, m.n_sel) == (8124, 1092)
    assert (w.n_cand, w.n_sel, w.first_new_block) == (32636, 2180, 32640)
    assert m.n_blocks * m.block == 262144 and w.n_blocks * w.block == 1 << 20


def test_token_inputs_deterministic_and_paged():
    w = synth.scaled(synth.TOKEN["8b"], L=2, N=512, turns=2, R=8)
    a, b = synth.token_inputs(w), synth.token_inputs(w)
    assert torch.equal(a["pool"], b["pool"]) and torch.equal(a["slot_map"], b["slot_map"])
    assert torch.equal(a["turns"], b["turns"])
    assert a["pool"].shape == (2, 512, 8, 128) and a["pool"].dtype == torch.bfloat16
    assert a["turns"].shape == (2, 2, 32, 8, 128)
    s = a["slot_map"].long()
    assert torch.equal(torch.sort(s).values, torch.arange(512))             # a bijection onto the pool
    pages = s.view(-1, w.page)
    assert torch.equal(pages - pages[:, :1], torch.arange(w.page).expand_as(pages))  # contiguous within a page
    assert torch.all(pages[:, 0] % w.page == 0)
    other = synth.token_inputs(dataclasses.replace(w, seed=w.seed + 1))
    assert not torch.equal(other["pool"], a["pool"])


def test_identity_map_and_fp32_for_tiny():
    x = synth.token_inputs(synth.TOKEN["tiny"])
    assert x["slot_map"] is None and x["pool"].dtype == torch.float32
    assert x["turns"].shape == (3, 2, 4, 16, 64)


def test_outlier_channels():
    w = synth.scaled(synth.TOKEN["long"], L=1, N=4096, turns=1, R=4)
    pool = synth.token_inputs(w)["pool"].float()                   # [1, N, Hkv, D]
    std = pool[0].std(dim=0)                                        # [Hkv, D]
    n_out = round(0.02 * w.D)
    for g in range(w.Hkv):
        big = (std[g] > 4.0).sum().item()
        assert big == n_out, (g, big)
        assert torch.allclose(std[g][std[g] > 4.0], torch.full((n_out,), 8.0), rtol=0.1)
        assert torch.allclose(std[g][std[g] <= 4.0], torch.ones(w.D - n_out), rtol=0.1)


def test_block_inputs_structure():
    w = synth.scaled(synth.BLOCK["ws1m"], L=1, Hq=5, Hkv=1, n_blocks=600, M=4, k=64, n_recent=8, new_tokens=64 * 32)
    x = synth.block_inputs(w)
    first = w.first_new_block
    assert first == 600 - 64
    assert x["raw"].shape == (1, 1, 64 * 32, 128)
    assert torch.count_nonzero(x["index"][:, :, first:]) == 0      # the new blocks are built by the step
    old = x["index"][0, 0, :first].float()
    # offset ~ N(0, 0.25) plus the spread of a 32-token mean, N(0, 1/32)
    assert abs(old.std().item() - (0.25 + 1 / 32) ** 0.5) < 0.02
    raw = x["raw"][0, 0].float().view(64, 32, 128)
    assert abs((raw - raw.mean(dim=1, keepdim=True)).std().item() - 1.0) < 0.02   # unit noise within a block
    assert abs(raw.mean(dim=1).std().item() - (0.25 + 1 / 32) ** 0.5) < 0.03     # block offsets
    assert torch.equal(torch.sort(x["page_perm"]).values, torch.arange(w.n_sel, dtype=torch.int32))
    assert x["staging"].shape == (1, 1, min(w.k, w.n_cand) * 32, 128)
    src, page, pos0 = synth.scatter_plan_incremental(w, x["page_perm"])
    assert torch.equal(pos0, (torch.arange(len(src), dtype=torch.int32) + w.n_sink) * w.block)
    assert torch.equal(page, x["page_perm"][(torch.arange(len(src)) + w.n_sink)])


def test_full_build_scatter_plan():
    w = synth.scaled(synth.BLOCK["meank262k"], L=1, Hq=5, Hkv=1, n_blocks=40, M=4, k=8, n_recent=4)
    x = synth.block_inputs(w)
    assert x["raw"].shape == (1, 1, 40 * 32, 128) and "staging" not in x
    page, pos0 = synth.scatter_plan_full(w, x["page_perm"])
    assert len(page) == w.n_sel and torch.equal(pos0, torch.arange(w.n_sel, dtype=torch.int32) * 32)


# ---------------------------------------------------------------------------
# platform-independent draws (inputs of the stored full-size oracle values)
# ---------------------------------------------------------------------------

def test_portable_draws_are_fixed():
    """The first draws of one key, as recorded on the host that wrote the stored oracle values
    (bf16 bit patterns): a change in numpy's PCG64 stream or normal sampler shows up here."""
    x = synth.portable_normal((6,), (1005, 4, 0))
    assert synth.bf16_bits(x).tolist() == [15906, 16161, 48408, 49002, 49057, 16242]


def test_portable_draws_spread_and_independence():
    import numpy as np
    a = synth.portable_normal((1 << 20,), (7, 1, 0)).astype(np.float64)
    b = synth.portable_normal((1 << 20,), (7, 1, 1)).astype(np.float64)
    assert abs(a.mean()) < 5e-3 and abs(a.std() - 1) < 5e-3
    assert abs(np.corrcoef(a, b)[0, 1]) < 5e-3       # another layer key: another stream
    s = synth.portable_normal((1 << 16,), (7, 1, 0), std=0.25)
    assert np.array_equal(s, a[:1 << 16].astype(np.float32) * np.float32(0.25))


def test_portable_block_layers():
    import numpy as np
    w = synth.scaled(synth.BLOCK["ws1m"], L=2, Hq=10, Hkv=2, n_blocks=64, M=8)
    x0, x0b, x1 = synth.portable_block_layer(w, 0), synth.portable_block_layer(w, 0), synth.portable_block_layer(w, 1)
    assert x0["q"].shape == (10, 8, 128) and x0["index"].shape == (2, 64, 128) and x0["q"].dtype == np.uint16
    assert synth.portable_layer_digest(x0) == synth.portable_layer_digest(x0b) != synth.portable_layer_digest(x1)
    # the workspace index spreads as offset + mean of a block: sigma^2 + 1/block
    big = synth.scaled(w, n_blocks=4096)
    v = (synth.portable_block_layer(big, 0)["index"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(v.std() - (0.25 + 1 / 32) ** 0.5) < 0.01
    # full build: raw K of a block shares one offset per channel
    m = synth.scaled(synth.BLOCK["meank262k"], L=1, Hq=5, Hkv=1, n_blocks=512, M=4)
    raw = (synth.portable_block_layer(m, 0)["raw"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    means = raw.reshape(1, 512, 32, 128).mean(axis=2)
    assert abs(means.std() - (0.25 + 1 / 32) ** 0.5) < 0.02 and abs(raw.std() - 1.25 ** 0.5) < 0.01
    d = synth.portable_digest([synth.portable_layer_digest(x0), synth.portable_layer_digest(x1)])
    assert len(d) == 64 and d != synth.portable_digest([synth.portable_layer_digest(x1), synth.portable_layer_digest(x0)])
