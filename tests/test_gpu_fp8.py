"""FP8 (E4M3) storage of the Mean-K index through the C ABI against the oracle:
codes, scale exponents and expanded rows bit for bit; R_b on the expanded index
within the score tolerance; host-side argument checks."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_scores_close, bits, f64

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = kv.Context(0)
    yield c
    c.close()


def _index(rng, rows, D):
    """Rows of mixed magnitude, with zero, signed-zero, tiny and huge rows and exact ties."""
    x = rng.standard_normal((rows, D)).astype(np.float32) * (10.0 ** rng.uniform(-6, 6, (rows, 1))).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2] = 1e-38
    x[3, :] = 3e38 * np.sign(rng.standard_normal(D))
    x[4, :4] = [448.0, 1.0625, 1.1875, -2.0 ** -10]       # exact ties in E4M3 (e = 0 for this row)
    x[4, 4:] = 0.5
    x[5] = rng.integers(-8, 8, D).astype(np.float32) * 2.0 ** -8
    return torch.from_numpy(x).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("rows,D", [(1, 128), (37, 128), (4099, 128), (301, 64), (65, 256)])
def test_fp8_index_bit_exact(ctx, rows, D):
    rng = np.random.default_rng(rows + D)
    idx = _index(rng, max(rows, 6), D)[:rows].contiguous()
    codes, exps = ctx.index_to_fp8(idx)
    back = ctx.index_from_fp8(codes, exps)
    ctx.check_device()
    ref_c, ref_e = oracle.index_to_fp8(bits(idx))
    assert np.array_equal(exps.cpu().numpy(), ref_e)
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(bits(back), oracle.index_from_fp8(ref_c, ref_e))


def test_fp8_index_every_code_expands_exactly(ctx):
    """All 254 finite codes at several exponents, through the GPU expansion."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    codes = np.resize(codes, 256).reshape(2, 128)
    for e in (-100, -9, 0, 7, 100):
        exps = np.full(2, e, np.int8)
        out = ctx.index_from_fp8(torch.from_numpy(codes).cuda(), torch.from_numpy(exps).cuda())
        ctx.check_device()
        assert np.array_equal(bits(out), oracle.index_from_fp8(codes, exps))


def test_fp8_index_full_size_sampled(ctx):
    """The 1M-token workspace's index (L64 Hkv8, 32768 blocks, D128): 16.8M rows, 4096 sampled
    against the oracle; every row's stored values within the format's error bound."""
    L, Hkv, nb, D = 64, 8, 32768, 128
    g = torch.Generator(device="cuda").manual_seed(7)
    idx = (torch.randn((L * Hkv * nb, D), device="cuda", generator=g) * 0.3).to(torch.bfloat16)
    codes, exps = ctx.index_to_fp8(idx)
    back = ctx.index_from_fp8(codes, exps)
    ctx.check_device()
    rng = np.random.default_rng(3)
    rows = torch.as_tensor(np.sort(rng.choice(idx.shape[0], 4096, replace=False)), device="cuda")
    ref_c, ref_e = oracle.index_to_fp8(bits(idx[rows]))
    assert np.array_equal(codes[rows].cpu().numpy(), ref_c)
    assert np.array_equal(exps[rows].cpu().numpy(), ref_e)
    # bound on all rows, in chunks: |back - x| <= 2^-4 |x| + 2^-10 * 2^e
    for r0 in range(0, idx.shape[0], 1 << 20):
        x, y = idx[r0:r0 + (1 << 20)].float(), back[r0:r0 + (1 << 20)].float()
        tol = x.abs() * 2.0 ** -4 + torch.exp2(exps[r0:r0 + (1 << 20)].float() - 10.0)[:, None]
        assert bool(((y - x).abs() <= tol).all())
    assert bool((exps.float() >= -100).all())


def test_block_scores_on_expanded_fp8_index(ctx):
    """R_b from the expanded FP8 index against the oracle's R_b on the oracle's expanded index."""
    rng = np.random.default_rng(11)
    L, Hq, Hkv, M, D, nb = 2, 8, 2, 300, 128, 700
    q = torch.from_numpy(rng.standard_normal((L, Hq, M, D)).astype(np.float32)).to(torch.bfloat16).cuda()
    ix = torch.from_numpy((rng.standard_normal((L, Hkv, nb, D)) * 0.5).astype(np.float32)).to(torch.bfloat16).cuda()
    codes, exps = ctx.index_to_fp8(ix)
    ix8 = ctx.index_from_fp8(codes, exps)
    R = torch.empty(nb, device="cuda")
    ctx.block_scores(q, ix8, nb, 4, 16, R)
    ctx.check_device()
    ref_c, ref_e = oracle.index_to_fp8(bits(ix))
    Rref = oracle.block_scores(bits(q), oracle.index_from_fp8(ref_c, ref_e), nb, 4, 16)
    assert_scores_close(f64(R), Rref, what="R_b on the FP8 index")
    # and how far the FP8 index moves R_b from the bf16 one (informative bound, not parity)
    R16 = oracle.block_scores(bits(q), bits(ix), nb, 4, 16)
    C = slice(4, nb - 16)
    assert np.max(np.abs(Rref[C] - R16[C]) / R16[C]) < 0.1


def test_fp8_index_argument_checks(ctx):
    idx = torch.zeros((4, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kv.KvselError):
        ctx.index_to_fp8(idx)                              # D = 96 unsupported
    idx = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    codes = torch.empty((4 * 128 + 1,), dtype=torch.uint8, device="cuda")[1:].view(4, 128)
    with pytest.raises(kv.KvselError):
        ctx.index_to_fp8(idx, codes=codes)                 # codes not 4-byte aligned
    empty = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    c0, e0 = ctx.index_to_fp8(empty)
    assert c0.numel() == 0 and e0.numel() == 0
