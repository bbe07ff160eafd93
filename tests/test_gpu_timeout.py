"""The tensor-core kernel's give-up path, driven without faulting or hanging the GPU.

Every mbarrier wait in the block scorer is bounded; when one gives up the CTA
flags KVSEL_ERR_TIMEOUT in the device error word, drains its own copies and
MMAs with bounded waits, frees its tensor memory and returns.  The internal
test entry kvsel_test_block_scores_give_up makes the row pass's first MMA
issuer wait on a barrier that nothing completes (with a 2 ms limit) while the
producer's copies and the other issuer's MMAs are in flight.  The call must
report the timeout, and the next normal call on the same context must run
green and match the oracle (tensor memory freed, barriers and workspace
usable)."""
import ctypes

import pytest
import torch

import oracle
from helpers import assert_scores_close, bits, f64

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402

_P, _I = ctypes.c_void_p, ctypes.c_int


@pytest.fixture(scope="module")
def give_up():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = kv._lib.kvsel_test_block_scores_give_up
    fn.restype = _I
    fn.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_uint64, _P]
    return fn


def _inputs(L, Hq, Hkv, M, Bcap, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((L, Hq, M, 128), generator=gen, device="cuda").to(torch.bfloat16)
    ix = (torch.randn((L, Hkv, Bcap, 128), generator=gen, device="cuda") * 0.5).to(torch.bfloat16)
    return q, ix


@pytest.mark.parametrize("L,Hq,Hkv,M,nb", [(1, 8, 2, 64, 1000), (2, 10, 2, 300, 2100)])
def test_block_scores_give_up_then_recover(give_up, L, Hq, Hkv, M, nb):
    ctx = kv.Context(0)
    S, Rc = 4, 16
    q, ix = _inputs(L, Hq, Hkv, M, nb, seed=nb)
    ref = oracle.block_scores(bits(q), bits(ix), nb, S, Rc)
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # twice in a row on the same context
        R = torch.full((nb,), float("nan"), device="cuda")
        rc = give_up(ctx.handle, q.data_ptr(), ix.data_ptr(), L, Hq, Hkv, M, 128, nb, nb, S, Rc, R.data_ptr(),
                     2_000_000, s)
        assert rc == kv.OK, kv.kvsel_last_error_string(ctx.handle)
        assert kv.kvsel_check_device(ctx.handle, s) == kv.ERR_TIMEOUT, kv.kvsel_last_error_string(ctx.handle)
        assert "gave up" in kv.kvsel_last_error_string(ctx.handle)
        # the next normal call on the same context is green and right
        R = torch.full((nb,), float("nan"), device="cuda")
        ctx.block_scores(q, ix, nb, S, Rc, R)
        ctx.check_device()
        assert_scores_close(f64(R), ref, what="R_b after a give-up")
    ctx.close()


def test_give_up_entry_rejects_bad_limits(give_up):
    ctx = kv.Context(0)
    q, ix = _inputs(1, 4, 1, 8, 64, seed=1)
    R = torch.zeros(64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for wait in (0, 2_000_000_000):
        rc = give_up(ctx.handle, q.data_ptr(), ix.data_ptr(), 1, 4, 1, 8, 128, 64, 64, 0, 0, R.data_ptr(), wait, s)
        assert rc == kv.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(R == 0)
    ctx.close()
