"""The single-session calls are asynchronous and, once their workspace has grown, do no
allocation or synchronisation, so a whole IntentKV step and a whole KVMEM step can be
captured in one CUDA graph and replayed.  The replay must give the eager results bit for bit
(every kernel of the two steps is deterministic)."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

import kv_cache_retention_gb300 as kv  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = kv.Context(0)
    yield c
    c.close()


def _token_step(ctx, w, t, M, rule, keep, keep_idx, slot_out):
    smap = t["slot_map"] if t["slot_map"] is not None else t["identity"]
    ctx.memory_update(t["q_last"], w.lam, M)
    ctx.rule_scores(t["pool"], M, w.L, w.Hq, w.Hkv, w.N, w.D, w.pi, w.q_s, w.q_e, rule, slot_map=t["slot_map"],
                    n_slots=w.N)
    ctx.topk_retain(rule, w.pi, w.q_s, w.q_e, w.C, keep=keep, keep_idx=keep_idx)
    ctx.redirect_slots(smap, keep, w.dead_slot, slot_out)


def _block_step(ctx, b, bi, R, ids, dst_page, dst_pos0):
    ctx.meank_build(bi["raw"], b.block, bi["index"])
    ctx.block_scores(bi["q"], bi["index"], b.n_blocks, b.n_sink, b.n_recent, R)
    ctx.select_blocks(R, b.n_sink, b.n_recent, b.k, ids)
    ctx.rerope_scatter(bi["raw"], ids, dst_page, dst_pos0, bi["pool"], b.rope_base)


@pytest.mark.parametrize("name", ["tiny", "8b"])
def test_token_step_replays_from_a_cuda_graph(ctx, name):
    w = synth.TOKEN[name]
    t = synth.token_inputs(w, "cuda")
    t["q_last"] = t["turns"][w.turns - 1].contiguous()
    t["identity"] = torch.arange(w.N, device="cuda", dtype=torch.int32)
    M0 = torch.nn.functional.normalize(torch.randn((w.L, w.Hq, w.D), device="cuda"), dim=-1)
    outs = [dict(M=M0.clone(), rule=torch.empty(w.N, device="cuda"),
                 keep=torch.empty(w.N, device="cuda", dtype=torch.uint8),
                 keep_idx=torch.zeros(w.N, device="cuda", dtype=torch.int32),
                 slot_out=torch.empty(w.N, device="cuda", dtype=torch.int32)) for _ in range(2)]
    e, gph = outs
    _token_step(ctx, w, t, **e)                      # eager (also grows the workspace)
    torch.cuda.synchronize()
    ctx.check_device()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                        # warm the capture stream
        gph["M"].copy_(M0)
        _token_step(ctx, w, t, **gph)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _token_step(ctx, w, t, **gph)
    for _ in range(3):
        gph["M"].copy_(M0)
        gph["rule"].fill_(-1.0)
        g.replay()
    torch.cuda.synchronize()
    ctx.check_device()
    for k in ("M", "rule", "keep", "keep_idx", "slot_out"):
        assert torch.equal(e[k], gph[k]), k


def test_block_step_replays_from_a_cuda_graph(ctx):
    b = synth.scaled(synth.BLOCK["meank262k"], L=2, Hq=10, Hkv=2, n_blocks=300, M=64, k=40, n_recent=8,
                     new_tokens=300 * 32)
    bi = synth.block_inputs(b, "cuda")
    dst_page, dst_pos0 = synth.scatter_plan_full(b, bi["page_perm"])
    R = [torch.empty(b.n_blocks, device="cuda") for _ in range(2)]
    ids = [torch.empty(b.n_sel, device="cuda", dtype=torch.int32) for _ in range(2)]
    _block_step(ctx, b, bi, R[0], ids[0], dst_page, dst_pos0)
    torch.cuda.synchronize()
    ctx.check_device()
    pool0, index0 = bi["pool"].clone(), bi["index"].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _block_step(ctx, b, bi, R[1], ids[1], dst_page, dst_pos0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _block_step(ctx, b, bi, R[1], ids[1], dst_page, dst_pos0)
    bi["pool"].zero_()
    bi["index"].zero_()
    R[1].fill_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    ctx.check_device()
    assert torch.equal(R[0], R[1]) and torch.equal(ids[0], ids[1])
    assert torch.equal(bi["index"], index0) and torch.equal(bi["pool"], pool0)
