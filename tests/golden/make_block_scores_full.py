"""Write the fp64 oracle's full-size block scores of the two block workloads.

    python tests/golden/make_block_scores_full.py [--procs P] [--only meank262k|ws1m]

Output: tests/golden/block_scores_full.npz with, for each workload,
  <name>_R        R_b over every block (fp64), the oracle's block_scores
  <name>_mass_lg  the sampled (layer, kv head) pairs
  <name>_mass     their unnormalised candidate mass rows (fp64)
  <name>_sha256   digest of the input bytes (synth.portable_digest)
and the wall time, process count and host of the run.

Only the oracle computes here.  The inputs come from synth's platform-
independent draws (synth.portable_block_layer), layer by layer, so a worker
draws exactly the layers it needs.  The unchanged single-threaded oracle runs
in P processes over disjoint (layer, kv head) slices; the parent adds the mass
rows in ascending (layer, kv head) order and divides by L*Hq, which is the
order and arithmetic of the oracle's own block_scores, so the stored vector
does not depend on P.  The Mean-K index of the full-build workload is the
oracle's own build of the drawn raw K.
"""
from __future__ import annotations

import argparse
import multiprocessing as mp
import os
import platform
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
OUT = os.path.join(HERE, "block_scores_full.npz")

# (layer, kv head) pairs whose mass rows are stored: both corners and six spread between
MASS_PAIRS = [(0, 0), (9, 3), (17, 5), (31, 1), (32, 6), (47, 2), (55, 4), (63, 7)]

_cache = {}


def _layer(w, l):
    import synth
    if _cache.get("key") != (w, l):
        _cache.clear()
        _cache["key"] = (w, l)
        _cache["layer"] = synth.portable_block_layer(w, l)
    return _cache["layer"]


def _task_full_build(wl):
    """Full-build workload: one layer's Mean-K index (oracle) and all its (l, g) mass rows."""
    import oracle
    import synth
    w, l = wl
    x = _layer(w, l)
    digest = synth.portable_layer_digest(x)
    index = oracle.meank_build(x["raw"][None], w.block)
    parts = np.stack([oracle.block_mass(x["q"][None], index, w.n_blocks, w.n_sink, w.n_recent, 0, g)
                      for g in range(w.Hkv)])
    return l, digest, parts


def _task_workspace(wlg):
    """Workspace workload: the mass row of one (l, g) on the drawn index."""
    import oracle
    import synth
    w, l, g = wlg
    x = _layer(w, l)
    digest = synth.portable_layer_digest(x) if g == 0 else None
    part = oracle.block_mass(x["q"][None], x["index"][None], w.n_blocks, w.n_sink, w.n_recent, 0, g)
    return l, g, digest, part


def _init():
    sys.path.insert(0, ROOT)
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import torch
    torch.set_num_threads(1)


def run(name, procs, w=None, pairs=MASS_PAIRS):
    """Oracle R_b (and the mass rows of `pairs`) of block workload `name` (or of `w`, a
    scaled copy of it) with `procs` worker processes."""
    sys.path.insert(0, ROOT)
    import synth
    w = synth.BLOCK[name] if w is None else w
    t0 = time.time()
    parts = {}
    digests = {}
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs, initializer=_init) as pool:
        if not w.incremental:
            for l, digest, p in pool.imap_unordered(_task_full_build, [(w, l) for l in range(w.L)]):
                digests[l] = digest
                for g in range(w.Hkv):
                    parts[(l, g)] = p[g]
                print(f"{name}: layer {l} done ({time.time() - t0:.0f} s)", flush=True)
        else:
            tasks = [(w, l, g) for l in range(w.L) for g in range(w.Hkv)]
            for i, (l, g, digest, p) in enumerate(pool.imap_unordered(_task_workspace, tasks)):
                if digest is not None:
                    digests[l] = digest
                parts[(l, g)] = p
                if i % 16 == 15:
                    print(f"{name}: {i + 1} of {len(tasks)} (layer, kv head) rows ({time.time() - t0:.0f} s)",
                          flush=True)
    R = np.zeros(w.n_blocks)
    for l in range(w.L):
        for g in range(w.Hkv):
            R += parts[(l, g)]
    R /= float(w.L) * float(w.Hq)
    out = {f"{name}_R": R,
           f"{name}_mass_lg": np.array(pairs, dtype=np.int32),
           f"{name}_mass": np.stack([parts[tuple(lg)] for lg in pairs]),
           f"{name}_sha256": np.array(synth.portable_digest([digests[l] for l in range(w.L)])),
           f"{name}_wall_s": np.array(time.time() - t0),
           f"{name}_procs": np.array(procs)}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--procs", type=int, default=max(1, (os.cpu_count() or 2) - 1))
    ap.add_argument("--only", choices=["meank262k", "ws1m"])
    args = ap.parse_args()
    stored = dict(np.load(OUT)) if os.path.exists(OUT) else {}
    for name in ("meank262k", "ws1m"):
        if args.only and name != args.only:
            continue
        stored.update(run(name, args.procs))
        stored["host"] = np.array(f"{platform.machine()} {platform.processor()} nproc={os.cpu_count()}")
        np.savez_compressed(OUT, **stored)
        print(f"{name}: written ({float(stored[name + '_wall_s']):.0f} s with {args.procs} processes)", flush=True)


if __name__ == "__main__":
    main()
