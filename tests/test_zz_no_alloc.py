"""kvsel_rule_scores_noalloc: the rule-score call for callers that cannot let a
library allocate device memory (engines that give the GPU to their own KV pool
and allocator, loops that cannot take cudaFree's device synchronisation).

It runs the same kernels as kvsel_rule_scores on a fixed scratch array inside
the library, so its scores must equal that call's bit for bit, call after call,
and both must match the oracle.  Its context never makes an allocating call,
and the device's free memory must not move while it runs.  Collected last on
purpose."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_scores_close, bits

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402
import synth  # noqa: E402


def _call(fn, ctx, w, inp, M, rule, n_slots=None):
    s = torch.cuda.current_stream().cuda_stream
    pool = inp["pool"]
    code = kv.BF16 if pool.dtype == torch.bfloat16 else kv.F32
    sm = inp["slot_map"]
    return fn(ctx.handle, pool.data_ptr(), code, None if sm is None else sm.data_ptr(), w.N if n_slots is None else n_slots,
              w.L, w.Hq, w.Hkv, w.N, w.D, w.N * w.Hkv * w.D, w.Hkv * w.D, M.data_ptr(), w.pi, w.q_s, w.q_e,
              rule.data_ptr(), s)


def _oracle(w, inp, M):
    pool = inp["pool"]
    k = bits(pool).ravel() if pool.dtype == torch.bfloat16 else pool.cpu().numpy().ravel()
    sm = None if inp["slot_map"] is None else inp["slot_map"].cpu().numpy()
    return oracle.rule_scores(k, M.cpu().double().numpy(), w.L, w.Hq, w.Hkv, w.N, w.D, w.pi, w.q_s, w.q_e,
                              slot_map=sm)


def test_noalloc_matches_rule_scores_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    small = synth.scaled(synth.TOKEN["8b"], L=4, N=4096, C=1024, span=256)
    cases = []
    for w, seed in [(synth.TOKEN["tiny"], 1), (small, 2)]:
        inp = synth.token_inputs(w, "cuda")
        gen = torch.Generator(device="cuda").manual_seed(seed)
        M = torch.nn.functional.normalize(torch.randn((w.L, w.Hq, w.D), generator=gen, device="cuda"), dim=-1)
        cases.append((w, inp, M, torch.full((w.N,), float("nan"), device="cuda"), torch.empty(w.N, device="cuda")))
    ctx = kv.Context(0)       # only ever used for the no-allocation call
    ref_ctx = kv.Context(0)   # the allocating call runs on its own context
    torch.cuda.synchronize()

    # the first call looks up the scratch array's address (and loads its module)
    w, inp, M, got, ref = cases[0]
    assert _call(kv.kvsel_rule_scores_noalloc, ctx, w, inp, M, got) == kv.OK, kv.kvsel_last_error_string(ctx.handle)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    # two calls in a row on different inputs: the shared scratch keeps the last
    # call's contents, which must not leak into the next result
    for w, inp, M, got, ref in cases:
        got.fill_(float("nan"))
        assert _call(kv.kvsel_rule_scores_noalloc, ctx, w, inp, M, got) == kv.OK, kv.kvsel_last_error_string(ctx.handle)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "device memory changed during kvsel_rule_scores_noalloc calls"
    for w, inp, M, got, ref in cases:
        assert _call(kv.kvsel_rule_scores, ref_ctx, w, inp, M, ref) == kv.OK, kv.kvsel_last_error_string(ref_ctx.handle)
    torch.cuda.synchronize()
    # the same kernels: bit-identical scores
    for w, inp, M, got, ref in cases:
        assert torch.equal(got, ref), f"noalloc {w.name}: differs from kvsel_rule_scores"
        want = _oracle(w, inp, M)
        assert_scores_close(got.cpu().double().numpy(), want, what=f"noalloc {w.name} vs oracle")
        assert_scores_close(ref.cpu().double().numpy(), want, what=f"rule_scores {w.name} vs oracle")
    # the measurement above can see an allocation: the allocating call grows the
    # workspace of a context that has none yet
    w, inp, M, got, ref = cases[1]
    assert _call(kv.kvsel_rule_scores, ctx, w, inp, M, ref) == kv.OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] < free0
    ctx.check_device()
    ref_ctx.check_device()
    ctx.close()
    ref_ctx.close()


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
