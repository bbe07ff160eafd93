"""kvsel_rule_scores_noalloc: the rule-score call for callers that cannot let a
library allocate device memory (engines that give the GPU to their own KV pool
and allocator, graph-recorded code, loops that cannot take cudaFree's device
synchronisation).  It must give the same scores as kvsel_rule_scores, call
after call, on its fixed scratch array.  Collected last on purpose."""
import pytest
import torch

from helpers import assert_scores_close

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402
from kv_cache_retention_gb300 import synth  # noqa: E402


def _call(fn, ctx, w, inp, M, rule, n_slots=None):
    s = torch.cuda.current_stream().cuda_stream
    pool = inp["pool"]
    code = kv.BF16 if pool.dtype == torch.bfloat16 else kv.F32
    sm = inp["slot_map"]
    return fn(ctx.handle, pool.data_ptr(), code, None if sm is None else sm.data_ptr(), w.N if n_slots is None else n_slots,
              w.L, w.Hq, w.Hkv, w.N, w.D, w.N * w.Hkv * w.D, w.Hkv * w.D, M.data_ptr(), w.pi, w.q_s, w.q_e,
              rule.data_ptr(), s)


def test_noalloc_matches_rule_scores_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx = kv.Context(0)
    # two calls in a row on different inputs: the shared scratch keeps the last
    # call's contents, which must not leak into the next result
    small = synth.scaled(synth.TOKEN["8b"], L=4, N=4096, C=1024, span=256)
    for w, seed in [(synth.TOKEN["tiny"], 1), (small, 2)]:
        inp = synth.token_inputs(w, "cuda")
        gen = torch.Generator(device="cuda").manual_seed(seed)
        M = torch.nn.functional.normalize(torch.randn((w.L, w.Hq, w.D), generator=gen, device="cuda"), dim=-1)
        ref = torch.empty(w.N, device="cuda")
        got = torch.full((w.N,), float("nan"), device="cuda")
        assert _call(kv.kvsel_rule_scores, ctx, w, inp, M, ref) == kv.OK, kv.kvsel_last_error_string(ctx.handle)
        assert _call(kv.kvsel_rule_scores_noalloc, ctx, w, inp, M, got) == kv.OK, kv.kvsel_last_error_string(ctx.handle)
        torch.cuda.synchronize()
        assert_scores_close(got.cpu().double().numpy(), ref.cpu().double().numpy(), what=f"noalloc {w.name}")
    ctx.check_device()
    ctx.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx = kv.Context(0)
    w = synth.TOKEN["8b"]  # 36*32*32768*4 bytes of logits: far beyond 64 MiB
    pool = torch.zeros((1,), device="cuda", dtype=torch.bfloat16)
    M = torch.zeros((w.L, w.Hq, w.D), device="cuda")
    rule = torch.full((w.N,), 3.0, device="cuda")
    rc = kv.kvsel_rule_scores_noalloc(ctx.handle, pool.data_ptr(), kv.BF16, None, w.N, w.L, w.Hq, w.Hkv, w.N, w.D,
                                      w.N * w.Hkv * w.D, w.Hkv * w.D, M.data_ptr(), w.pi, w.q_s, w.q_e,
                                      rule.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == kv.ERR_UNSUPPORTED
    assert "scratch" in kv.kvsel_last_error_string(ctx.handle)
    torch.cuda.synchronize()
    assert torch.all(rule == 3.0)
    ctx.close()
