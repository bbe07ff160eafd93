"""Host-side validation: every C-ABI call rejects bad arguments with the right
status, launches nothing and leaves its outputs untouched."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = kv.Context(0)
    yield c
    c.close()


def test_rule_scores_rejections(ctx):
    h = ctx.handle
    pool = torch.zeros((2, 64, 2, 64), device="cuda", dtype=torch.bfloat16)
    M = torch.zeros((2, 4, 64), device="cuda")
    rule = torch.full((64,), 5.0, device="cuda")
    p, m, r = pool.data_ptr(), M.data_ptr(), rule.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    f = kv.kvsel_rule_scores
    assert f(h, p, kv.BF16, None, 64, 2, 4, 2, 64, 64, 64 * 128, 128, m, 0, 64, 64, r, s) == kv.OK
    torch.cuda.synchronize()
    rule.fill_(5.0)
    assert f(h, None, kv.BF16, None, 64, 2, 4, 2, 64, 64, 64 * 128, 128, m, 0, 64, 64, r, s) == kv.ERR_INVALID_ARG
    assert f(h, p, 7, None, 64, 2, 4, 2, 64, 64, 64 * 128, 128, m, 0, 64, 64, r, s) == kv.ERR_INVALID_ARG
    assert f(h, p, kv.BF16, None, 64, 2, 5, 2, 64, 64, 64 * 128, 128, m, 0, 64, 64, r, s) == kv.ERR_SHAPE
    assert f(h, p, kv.BF16, None, 64, 2, 4, 2, 64, 48, 64 * 128, 128, m, 0, 64, 64, r, s) == kv.ERR_UNSUPPORTED
    assert f(h, p, kv.BF16, None, 64, 2, 4, 2, 64, 64, 64 * 128, 128, m, 0, 65, 64, r, s) == kv.ERR_SHAPE
    assert f(h, p, kv.BF16, None, 64, 2, 4, 2, 64, 64, 64 * 128, 128, m, 65, 0, 64, r, s) == kv.ERR_SHAPE
    assert f(h, p, kv.BF16, None, 10, 2, 4, 2, 64, 64, 64 * 128, 128, m, 0, 64, 64, r, s) == kv.ERR_SHAPE
    assert f(h, p + 2, kv.BF16, None, 64, 2, 4, 2, 64, 64, 64 * 128, 128, m, 0, 64, 64, r, s) == kv.ERR_ALIGN
    assert f(h, p, kv.BF16, None, 64, 2, 4, 2, 64, 64, 64 * 128 + 3, 128, m, 0, 64, 64, r, s) == kv.ERR_ALIGN
    assert f(h, p, kv.BF16, None, 64, 2, 36, 2, 64, 64, 64 * 128, 128, m, 0, 64, 64, r, s) == kv.ERR_UNSUPPORTED
    assert "Hq" in kv.kvsel_last_error_string(h) or "group" in kv.kvsel_last_error_string(h)
    torch.cuda.synchronize()
    assert torch.all(rule == 5.0)


def test_other_calls_reject(ctx):
    h = ctx.handle
    s = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(256, device="cuda")
    n = ctypes.c_int(-1)
    assert kv.kvsel_topk_retain(h, x.data_ptr(), 256, 0, 10, 5, 3, None, None, ctypes.byref(n), s) == kv.ERR_INVALID_ARG
    assert kv.kvsel_topk_retain(h, x.data_ptr(), 256, 0, 10, 5, 3, x.data_ptr(), None, ctypes.byref(n), s) == kv.ERR_SHAPE
    assert kv.kvsel_memory_update(h, x.data_ptr(), kv.F32, 1, 1, 1, 6, 0.5, 1, 0, x.data_ptr(), None, s) == kv.ERR_UNSUPPORTED
    assert kv.kvsel_memory_update(h, x.data_ptr(), kv.F32, 1, 1, 1, 8, -1.0, 1, 0, x.data_ptr(), None, s) == kv.ERR_INVALID_ARG
    assert kv.kvsel_memory_update(h, x.data_ptr(), kv.F32, 1, 1, 1, 8, 0.5, 1, 1, x.data_ptr(), None, s) == kv.ERR_INVALID_ARG
    assert kv.kvsel_meank_build(h, x.data_ptr(), 1, 1, 64, 128, 32, 0, None, 1e6, 0, x.data_ptr(), 1, s) == kv.ERR_SHAPE
    assert kv.kvsel_meank_build(h, x.data_ptr(), 1, 1, 64, 96, 32, 0, None, 1e6, 0, x.data_ptr(), 4, s) == kv.ERR_UNSUPPORTED
    assert kv.kvsel_block_scores(h, x.data_ptr(), x.data_ptr(), 1, 2, 1, 1, 64, 4, 4, 0, 0, x.data_ptr(), None, s) == kv.ERR_UNSUPPORTED
    assert kv.kvsel_block_scores(h, x.data_ptr(), x.data_ptr(), 1, 3, 2, 1, 128, 4, 4, 0, 0, x.data_ptr(), None, s) == kv.ERR_SHAPE
    assert kv.kvsel_block_scores(h, x.data_ptr(), x.data_ptr(), 1, 2, 1, 1, 128, 8, 4, 0, 0, x.data_ptr(), None, s) == kv.ERR_SHAPE
    assert kv.kvsel_select_blocks(h, x.data_ptr(), 10, -1, 0, 2, x.data_ptr(), ctypes.byref(n), s) == kv.ERR_SHAPE
    assert kv.kvsel_rerope_scatter(h, x.data_ptr(), 0, 0, 0, x.data_ptr(), x.data_ptr(), x.data_ptr(), 1, 1, 1, 64, 8,
                                   1e4, 5, x.data_ptr(), 1, s) == kv.ERR_INVALID_ARG
    assert kv.kvsel_rerope_scatter(h, x.data_ptr(), 0, 0, 0, x.data_ptr(), x.data_ptr(), x.data_ptr(), 1, 1, 1, 64, 8,
                                   0.5, 0, x.data_ptr(), 1, s) == kv.ERR_INVALID_ARG
    assert kv.kvsel_redirect_slots(h, None, x.data_ptr(), 4, 0, x.data_ptr(), s) == kv.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(x == 0)


def test_closed_form_counts(ctx):
    x = torch.zeros(1000, device="cuda")
    keep = torch.empty(1000, device="cuda", dtype=torch.uint8)
    assert ctx.topk_retain(x, 100, 50, 200, 300, keep=keep) == 300      # F=[0,200): C*=100
    assert ctx.topk_retain(x, 100, 50, 200, 50, keep=keep) == 200       # C < |F|: F only
    assert ctx.topk_retain(x, 0, 1000, 1000, 5000, keep=keep) == 1000   # N <= C
    ids = torch.empty(1000, device="cuda", dtype=torch.int32)
    assert ctx.select_blocks(x, 4, 64, 10000, ids) == 1000
    assert ctx.select_blocks(x, 600, 600, 3, ids) == 1000
