"""Seeded synthetic inputs for the retention path.

This module holds the workload definitions and the random input generators
that both the CUDA path and the fp64 oracle consume (the same bytes go to
both).  It contains none of the method's arithmetic: only random draws,
offsets, permutations and dtype casts.

Workloads (sizes from the pages' settings; no dataset or model weights are
used anywhere):
  token-level rule scoring (IntentKV):
    tiny   L2 Hq4 Hkv2 D64 N2048, fp32 K, identity slot map
    8b     L36 Hq32 Hkv8 D128 N32768, bf16 K, 16-slot pages shuffled
    long   L48 Hq40 Hkv8 D128 N92160, bf16 K with 2% outlier channels x8
  block retrieval (KVMEM):
    meank262k   L64 Hq40 Hkv8 D128, 262144 raw tokens = 8192 blocks of 32, M=512
    ws1m        L64 Hq40 Hkv8 D128, 32768 indexed blocks (1M-token workspace),
                4096 new tokens, M=2048, 2048 staged top blocks

Post-RoPE K for the rule scorer is drawn directly: a rotation of an i.i.d.
N(0,1) pair is again an i.i.d. N(0,1) pair, so RoPE(N(0,1)) and N(0,1) have the
same distribution and no rotation is needed here.  The "long" workload scales
2% of the channels of each (layer, kv head) of that post-RoPE K by 8.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class TokenWorkload:
    name: str
    L: int
    Hq: int
    Hkv: int
    D: int
    N: int
    dtype: str          # "f32" | "bf16"
    turns: int          # QueryMemory turns before scoring
    R: int              # query rows per turn (actionable span length)
    lam: float
    pi: int             # protected prefix length
    span: int           # current query span = the last `span` tokens
    C: int              # retention budget
    page: int           # slot-map page size; 0 = identity map
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    seed: int = 0

    @property
    def q_s(self):
        return self.N - self.span

    @property
    def q_e(self):
        return self.N

    @property
    def n_forced(self):
        lo, hi = self.q_s, min(self.q_e, self.pi)
        return self.pi + self.span - max(0, hi - lo)

    @property
    def n_cand(self):
        return self.N - self.n_forced

    @property
    def n_keep(self):
        return self.n_forced + min(max(0, self.C - self.n_forced), self.n_cand)

    @property
    def dead_slot(self):
        return self.N  # one past the pool

    def k_bytes(self):
        return self.L * self.N * self.Hkv * self.D * (2 if self.dtype == "bf16" else 4)


@dataclass(frozen=True)
class BlockWorkload:
    name: str
    L: int
    Hq: int
    Hkv: int
    D: int
    n_blocks: int       # indexed blocks after this step
    block: int          # tokens per block (= page size of the pool)
    M: int              # query tokens
    n_sink: int
    n_recent: int
    k: int              # top blocks by R_b
    new_tokens: int     # raw tokens whose blocks are (re)built this step
    incremental: bool   # False: the index is built from all raw tokens
    offset_sigma: float = 0.5
    rope_base: float = 1e6
    seed: int = 0

    @property
    def n_cand(self):
        return max(0, self.n_blocks - self.n_sink - self.n_recent)

    @property
    def n_sel(self):
        return self.n_sink + self.n_recent + min(self.k, self.n_cand)

    @property
    def first_new_block(self):
        return self.n_blocks - self.new_tokens // self.block


TOKEN = {
    "tiny": TokenWorkload("tiny L2 Hq4 Hkv2 D64 N2048 fp32", 2, 4, 2, 64, 2048, "f32", 3, 16, 0.5, 64, 128, 512, 0,
                          seed=1001),
    "8b": TokenWorkload("8B-shaped L36 Hq32 Hkv8 D128 N32768 bf16", 36, 32, 8, 128, 32768, "bf16", 5, 256, 0.3, 256,
                        512, 8192, 16, seed=1002),
    "long": TokenWorkload("long L48 Hq40 Hkv8 D128 N92160 bf16 outliers", 48, 40, 8, 128, 92160, "bf16", 12, 256, 0.3,
                          256, 1024, 8192, 16, outlier_frac=0.02, outlier_scale=8.0, seed=1003),
}

BLOCK = {
    "meank262k": BlockWorkload("Mean-K L64 Hq40 Hkv8 D128 262144 tokens (8192 blocks) M512", 64, 40, 8, 128, 8192, 32,
                               512, 4, 64, 1024, 262144, False, seed=1004),
    "ws1m": BlockWorkload("1M workspace L64 Hq40 Hkv8 D128 32768 blocks M2048", 64, 40, 8, 128, 32768, 32, 2048, 4, 128,
                          2048, 4096, True, seed=1005),
}


def scaled(w, **kw):
    """A copy of workload w with some sizes replaced (for parity cases)."""
    return dataclasses.replace(w, **kw)


def _gen(seed, device):
    return torch.Generator(device=device).manual_seed(int(seed))


def _bf16_or_f32(x, dtype):
    return x.to(torch.bfloat16) if dtype == "bf16" else x.float()


# ---------------------------------------------------------------------------
# token-level inputs
# ---------------------------------------------------------------------------

def token_inputs(w: TokenWorkload, device="cpu"):
    """Pool [L][N][Hkv][D], slot map [N] int32 or None, query turns [T][L][Hq][R][D]."""
    g = _gen(w.seed, device)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    pool = torch.empty((w.L, w.N, w.Hkv, w.D), dtype=dt, device=device)
    n_out = int(round(w.outlier_frac * w.D))
    for l in range(w.L):
        x = torch.randn((w.N, w.Hkv, w.D), generator=g, device=device)
        if n_out > 0:
            pick = torch.rand((w.Hkv, w.D), generator=g, device=device).argsort(dim=1)[:, :n_out]
            scale = torch.ones((w.Hkv, w.D), device=device)
            scale.scatter_(1, pick, w.outlier_scale)
            x = x * scale
        pool[l] = x.to(dt)
    slot_map = None
    if w.page > 0:
        n_pages = (w.N + w.page - 1) // w.page
        perm = torch.randperm(n_pages, generator=g, device=device).to(torch.int64)
        j = torch.arange(w.N, device=device)
        slot_map = (perm[j // w.page] * w.page + j % w.page).to(torch.int32)
        # the pool rows are i.i.d., so drawing them at slot positions is the same
        # as drawing per token and scattering through the slot map
    turns = torch.empty((w.turns, w.L, w.Hq, w.R, w.D), dtype=dt, device=device)
    for t in range(w.turns):
        turns[t] = torch.randn((w.L, w.Hq, w.R, w.D), generator=g, device=device).to(dt)
    return {"pool": pool, "slot_map": slot_map, "turns": turns}


# ---------------------------------------------------------------------------
# block-level inputs
# ---------------------------------------------------------------------------

def block_inputs(w: BlockWorkload, device="cpu", with_staging=True):
    """Raw K / index / queries / pool / page table for a block workload.

    full build (incremental=False): raw [L][Hkv][n_blocks*block][D] = per-block
      offset ~ N(0, sigma^2) + N(0,1) noise; the index is built from it.
    incremental: index blocks [0, first_new_block) are drawn directly as
      offset + N(0, 1/block) (the spread of a mean of `block` unit normals);
      raw [L][Hkv][new_tokens][D] = offset + N(0,1) for the new blocks; the
      staging buffer [L][Hkv][k*block][D] holds N(0,1) raw K of the top blocks.
    """
    g = _gen(w.seed, device)
    L, Hkv, D, blk = w.L, w.Hkv, w.D, w.block
    bf = torch.bfloat16
    out = {}
    n_raw_blocks = w.n_blocks if not w.incremental else w.new_tokens // blk
    raw = torch.empty((L, Hkv, n_raw_blocks * blk, D), dtype=bf, device=device)
    for l in range(L):
        off = torch.randn((Hkv, n_raw_blocks, 1, D), generator=g, device=device) * w.offset_sigma
        noise = torch.randn((Hkv, n_raw_blocks, blk, D), generator=g, device=device)
        raw[l] = (off + noise).reshape(Hkv, n_raw_blocks * blk, D).to(bf)
    out["raw"] = raw
    index = torch.zeros((L, Hkv, w.n_blocks, D), dtype=bf, device=device)
    if w.incremental:
        n_old = w.first_new_block
        for l in range(L):
            off = torch.randn((Hkv, n_old, D), generator=g, device=device) * w.offset_sigma
            noise = torch.randn((Hkv, n_old, D), generator=g, device=device) * (1.0 / blk) ** 0.5
            index[l, :, :n_old] = (off + noise).to(bf)
    out["index"] = index
    q = torch.empty((L, w.Hq, w.M, D), dtype=bf, device=device)
    for l in range(L):
        q[l] = torch.randn((w.Hq, w.M, D), generator=g, device=device).to(bf)
    out["q"] = q
    n_pages = w.n_sel
    out["page_perm"] = torch.randperm(n_pages, generator=g, device=device).to(torch.int32)
    out["pool"] = torch.zeros((L, n_pages, blk, Hkv, D), dtype=bf, device=device)
    if w.incremental and with_staging:
        n_top = min(w.k, w.n_cand)
        st = torch.empty((L, Hkv, n_top * blk, D), dtype=bf, device=device)
        for l in range(L):
            st[l] = torch.randn((Hkv, n_top * blk, D), generator=g, device=device).to(bf)
        out["staging"] = st
    return out


def scatter_plan_incremental(w: BlockWorkload, page_perm):
    """Entries of the staged top blocks: staging block i -> compact rank n_sink+i.

    The sink blocks come first in the ascending working set and the recent
    blocks last, so the i-th staged top block always has rank n_sink + i."""
    n_top = min(w.k, w.n_cand)
    i = torch.arange(n_top, device=page_perm.device, dtype=torch.int32)
    src_block = i
    rank = i + min(w.n_sink, w.n_blocks)
    dst_page = page_perm[rank.long()].to(torch.int32)
    dst_pos0 = (rank * w.block).to(torch.int32)
    return src_block, dst_page, dst_pos0


def scatter_plan_full(w: BlockWorkload, page_perm):
    """Destination of working-set entry r (ascending ids): page page_perm[r], position r*block."""
    r = torch.arange(w.n_sel, device=page_perm.device, dtype=torch.int32)
    return page_perm[r.long()].to(torch.int32), (r * w.block).to(torch.int32)


# ---------------------------------------------------------------------------
# platform-independent draws (inputs of the stored full-size oracle values)
# ---------------------------------------------------------------------------
# The stored fp64 block scores of the two block workloads are computed once on
# one host and compared on another (an x86 host writes them, the Arm host of the
# GPU reads them).  torch's CPU normal sampler is not the same on both: its
# vectorised Box-Muller path calls different transcendental implementations per
# instruction set.  numpy's PCG64 stream, seeded through SeedSequence, is
# defined bit for bit, and its float32 ziggurat normal sampler uses table
# lookups and IEEE arithmetic except in its rare tail and wedge branches, so a
# seed gives the same float32 draws on both hosts.  Every draw is keyed by
# (seed, tensor kind, layer) so that layers can be drawn in any order and in
# parallel.  A SHA-256 over the bf16 bytes, layer by layer, is recorded with the
# stored values and checked wherever they are used.

PORTABLE_RAW_OFFSET, PORTABLE_RAW_NOISE, PORTABLE_Q, PORTABLE_INDEX = 1, 2, 3, 4


def portable_normal(shape, key, std=1.0):
    """float32 N(0, std^2) draws from numpy's PCG64 seeded with the integer tuple `key`."""
    import numpy as np
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))
    x = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def bf16_bits(x):
    """float32 numpy array -> bf16 bit patterns (uint16), round to nearest even (torch's cast)."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def portable_block_layer(w: BlockWorkload, l: int):
    """Layer l of a block workload's inputs, as bf16 bit patterns (numpy uint16).

    Returns {"q": [Hq][M][D], and "raw": [Hkv][n_blocks*block][D] (full build: per
    (kv head, block, channel) offset ~ N(0, sigma^2) shared by the block's tokens,
    plus N(0,1) per token) or "index": [Hkv][n_blocks][D] (incremental workspace:
    every indexed block drawn directly as N(0, sigma^2 + 1/block), the spread of
    an offset plus the mean of `block` unit normals)}."""
    out = {"q": bf16_bits(portable_normal((w.Hq, w.M, w.D), (w.seed, PORTABLE_Q, l)))}
    if w.incremental:
        std = (w.offset_sigma ** 2 + 1.0 / w.block) ** 0.5
        out["index"] = bf16_bits(portable_normal((w.Hkv, w.n_blocks, w.D), (w.seed, PORTABLE_INDEX, l), std))
    else:
        off = portable_normal((w.Hkv, w.n_blocks, 1, w.D), (w.seed, PORTABLE_RAW_OFFSET, l), w.offset_sigma)
        noise = portable_normal((w.Hkv, w.n_blocks, w.block, w.D), (w.seed, PORTABLE_RAW_NOISE, l))
        noise += off
        out["raw"] = bf16_bits(noise.reshape(w.Hkv, w.n_blocks * w.block, w.D))
    return out


def portable_layer_digest(layer):
    """SHA-256 (hex) of one layer's bf16 bytes: q, then raw or index."""
    import hashlib
    h = hashlib.sha256()
    h.update(layer["q"].tobytes())
    h.update((layer["raw"] if "raw" in layer else layer["index"]).tobytes())
    return h.hexdigest()


def portable_digest(layer_digests):
    """SHA-256 (hex) over the per-layer digests in layer order."""
    import hashlib
    return hashlib.sha256("".join(layer_digests).encode()).hexdigest()
