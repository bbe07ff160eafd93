"""Checkpoint and resume: the only state a session carries between calls is
caller-owned device memory, the QueryMemory M [L][Hq][D] (IntentKV Sec. 3.2,
Eq. 2) and the Mean-K index (KVMEM "design and trade-offs" section).  Copying
either to the host and back into fresh buffers, on a fresh context, continues
the session bit for bit.  Also: NVTX ranges (KVSEL_NVTX=1) change no result."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402
import synth  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _token_turn(ctx, w, inp, M, t):
    ctx.memory_update(inp["turns"][t], w.lam, M, first_turn=(t == 0))
    rule = torch.empty(w.N, device="cuda")
    ctx.rule_scores(inp["pool"], M, w.L, w.Hq, w.Hkv, w.N, w.D, w.pi, w.q_s, w.q_e, rule, slot_map=inp["slot_map"],
                    n_slots=w.N)
    return rule


def test_query_memory_resume(gpu):
    w = synth.scaled(synth.TOKEN["8b"], L=4, N=4096, C=1024, span=256, turns=4, R=32)
    inp = synth.token_inputs(w, "cuda")
    a = kv.Context(0)
    M = torch.zeros((w.L, w.Hq, w.D), device="cuda")
    for t in range(w.turns - 1):
        _token_turn(a, w, inp, M, t)
    saved = M.cpu().clone()                                 # checkpoint after turn 3 of 4
    rule_a = _token_turn(a, w, inp, M, w.turns - 1)
    M_a = M.clone()
    torch.cuda.synchronize()
    a.close()
    b = kv.Context(0)                                       # resume elsewhere
    M2 = torch.empty((w.L, w.Hq, w.D), device="cuda")
    M2.copy_(saved)
    rule_b = _token_turn(b, w, inp, M2, w.turns - 1)
    torch.cuda.synchronize()
    b.check_device()
    assert torch.equal(M2, M_a) and torch.equal(rule_b, rule_a)
    b.close()


def test_meank_index_resume(gpu):
    w = synth.scaled(synth.BLOCK["ws1m"], L=2, Hq=10, Hkv=2, n_blocks=600, M=40, k=64, n_recent=8, new_tokens=64 * 32)
    inp = synth.block_inputs(w, "cuda", with_staging=False)
    a = kv.Context(0)
    index = inp["index"]
    a.meank_build(inp["raw"], w.block, index, first_block=w.first_new_block)
    R_a = torch.empty(w.n_blocks, device="cuda")
    a.block_scores(inp["q"], index, w.n_blocks, w.n_sink, w.n_recent, R_a)
    saved = index.cpu().clone()
    torch.cuda.synchronize()
    a.close()
    b = kv.Context(0)
    index2 = torch.empty_like(index)
    index2.copy_(saved)
    R_b = torch.empty(w.n_blocks, device="cuda")
    b.block_scores(inp["q"], index2, w.n_blocks, w.n_sink, w.n_recent, R_b)
    torch.cuda.synchronize()
    b.check_device()
    assert torch.equal(R_a, R_b)
    b.close()


_PROG = """
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
import kv_cache_retention_gb300 as kv, synth
w = synth.TOKEN["tiny"]
inp = synth.token_inputs(w, "cuda")
ctx = kv.Context(0)
M = torch.zeros((w.L, w.Hq, w.D), device="cuda")
for t in range(w.turns):
    ctx.memory_update(inp["turns"][t], w.lam, M, first_turn=(t == 0))
rule = torch.empty(w.N, device="cuda")
ctx.rule_scores(inp["pool"], M, w.L, w.Hq, w.Hkv, w.N, w.D, w.pi, w.q_s, w.q_e, rule)
ctx.check_device()
np.save(sys.argv[1], rule.cpu().numpy())
"""


def test_nvtx_ranges_change_nothing(gpu, tmp_path):
    outs = []
    for flag in ("0", "1"):
        path = str(tmp_path / f"rule_{flag}.npy")
        env = dict(os.environ, KVSEL_NVTX=flag)
        r = subprocess.run([sys.executable, "-c", _PROG.format(root=ROOT), path], env=env, capture_output=True,
                           text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(np.load(path))
    assert np.array_equal(outs[0], outs[1])
