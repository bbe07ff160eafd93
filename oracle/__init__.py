"""fp64 CPU oracle for the KV retention scoring / selection path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports this package, and this package never imports the product: the C source
``kvsel_oracle.c`` is compiled on its own with the host C compiler.

Every function takes numpy arrays.  bf16 tensors travel as ``uint16`` arrays of
their bit patterns; they are widened exactly inside the C code.  All arithmetic
is fp64.

The pins that tie this oracle to the pages (closed forms, invariants,
hand-worked examples, brute force) live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvsel_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")

F32 = 0
BF16 = 1
ROPE_NEOX = 0
ROPE_INTERLEAVED = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no fast-math: IEEE fp64)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            I64 = ctypes.c_int64
            D = ctypes.c_double
            lib.orc_double_to_bf16.argtypes = [D]
            lib.orc_double_to_bf16.restype = ctypes.c_uint16
            lib.orc_bf16_bits_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_bits_to_double.restype = D
            lib.orc_rope_rotate.argtypes = [P, I, D, D, I, I]
            lib.orc_memory_update.argtypes = [P, I, I, I, I, I, D, I, I, P, P]
            lib.orc_rule_scores.argtypes = [P, I, P, I, I, I, I, I, I64, I64, P, I, I, I, P]
            lib.orc_topk_retain.argtypes = [P, I, I, I, I, I, P, P]
            lib.orc_topk_retain.restype = I
            lib.orc_redirect_slots.argtypes = [P, P, I, ctypes.c_int32, P]
            lib.orc_meank_build.argtypes = [P, I, I, I, I, I, I, P, D, I, P, I, P]
            lib.orc_block_mass.argtypes = [P, P, I, I, I, I, I, I, I, I, I, I, I, P]
            lib.orc_block_scores.argtypes = [P, P, I, I, I, I, I, I, I, I, I, P, P]
            lib.orc_select_blocks.argtypes = [P, I, I, I, I, P]
            lib.orc_select_blocks.restype = I
            lib.orc_rerope_scatter.argtypes = [P, I64, I64, P, P, P, I, I, I, I, I, D, I, P, I]
            lib.orc_workset_diff.argtypes = [P, P, I, P, I, I, I, P, P, P, P, P, P, P, P]
            lib.orc_workset_diff.restype = I
            lib.orc_restore_blocks.argtypes = [P, P, I64, I64, P, P, P, I, I, I, I, I, D, I, P, P, I]
            lib.orc_rerope_shift.argtypes = [P, I, P, P, I, I, I, I, I, D, I]
            lib.orc_span_keep.argtypes = [P, P, I, P, I, P, I, P]
            lib.orc_span_keep.restype = I
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint]
            lib.orc_e4m3_decode.restype = D
            lib.orc_e4m3_encode.argtypes = [D]
            lib.orc_e4m3_encode.restype = ctypes.c_uint
            lib.orc_fp8_row_exp.argtypes = [P, I]
            lib.orc_fp8_row_exp.restype = I
            lib.orc_index_to_fp8.argtypes = [P, I64, I, P, P]
            lib.orc_index_from_fp8.argtypes = [P, P, I64, I, P]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dtype_code(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs are float32 or bf16 bits (uint16), got {a.dtype}")


# --------------------------------------------------------------------------
# element helpers
# --------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """fp64 -> bf16 bits, round to nearest even (one rounding)."""
    lib = _load()
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in, flat_out = x.ravel(), out.ravel()
    for i in range(flat_in.size):
        flat_out[i] = lib.orc_double_to_bf16(float(flat_in[i]))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bits -> fp64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rope_rotate(x, pos, base, style=ROPE_NEOX, inverse=False) -> np.ndarray:
    """Rotate one D-vector by RoPE at position ``pos`` (fp64)."""
    lib = _load()
    v = np.array(x, dtype=np.float64, copy=True)
    lib.orc_rope_rotate(_ptr(v), v.shape[-1], float(pos), float(base), int(style), int(bool(inverse)))
    return v


# --------------------------------------------------------------------------
# IntentKV
# --------------------------------------------------------------------------

def memory_update(q_rows, lam, M=None, first_turn=False, norm_mode=0, A=None):
    """One QueryMemory turn.  q_rows: [L,Hq,R,D] float32 or bf16 bits.

    Returns (M, A) as new fp64 arrays (A is None for norm_mode 0)."""
    lib = _load()
    q = np.ascontiguousarray(q_rows)
    L, Hq, R, D = q.shape
    M = np.zeros((L, Hq, D)) if M is None else np.array(M, dtype=np.float64, copy=True)
    if norm_mode != 0:
        A = np.zeros((L, Hq, D)) if A is None else np.array(A, dtype=np.float64, copy=True)
    lib.orc_memory_update(_ptr(q), _dtype_code(q), L, Hq, R, D, float(lam), int(bool(first_turn)),
                          int(norm_mode), _ptr(M), _ptr(A) if norm_mode != 0 else None)
    return M, (A if norm_mode != 0 else None)


def rule_scores(k_pool, M, L, Hq, Hkv, N, D, pi, q_s, q_e, slot_map=None,
                layer_stride=None, slot_stride=None):
    """IntentKV rule_j over N positions.  k_pool: flat float32 or bf16 bits."""
    lib = _load()
    k = np.ascontiguousarray(k_pool).ravel()
    Mm = _c(M, np.float64)
    sm = None if slot_map is None else _c(slot_map, np.int32)
    if slot_stride is None:
        slot_stride = Hkv * D
    if layer_stride is None:
        layer_stride = N * slot_stride
    rule = np.zeros(N, dtype=np.float64)
    lib.orc_rule_scores(_ptr(k), _dtype_code(k), _ptr(sm), L, Hq, Hkv, N, D, int(layer_stride),
                        int(slot_stride), _ptr(Mm), pi, q_s, q_e, _ptr(rule))
    return rule


def topk_retain(score, pi, q_s, q_e, C):
    """Eq. 1 keep set: returns (keep uint8 [N], keep_idx int32 ascending)."""
    lib = _load()
    s = _c(score, np.float64)
    N = s.size
    keep = np.zeros(N, dtype=np.uint8)
    idx = np.zeros(max(N, 1), dtype=np.int32)
    n = lib.orc_topk_retain(_ptr(s), N, pi, q_s, q_e, C, _ptr(keep), _ptr(idx))
    return keep, idx[:n].copy()


def redirect_slots(slot_in, keep, dead_slot):
    lib = _load()
    si = _c(slot_in, np.int32)
    kp = _c(keep, np.uint8)
    out = np.empty_like(si)
    lib.orc_redirect_slots(_ptr(si), _ptr(kp), si.size, int(dead_slot), _ptr(out))
    return out


# --------------------------------------------------------------------------
# KVMEM
# --------------------------------------------------------------------------

def meank_build(k_src, block, index=None, Bcap=None, first_block=0, src_pos=None,
                rope_base=1e6, rope_style=ROPE_NEOX, return_mean=False):
    """Mean-K of bf16 k_src [L,Hkv,T,D] into index bf16 bits [L,Hkv,Bcap,D]."""
    lib = _load()
    k = _c(k_src, np.uint16)
    L, Hkv, T, D = k.shape
    nb = (T + block - 1) // block
    if Bcap is None:
        Bcap = first_block + nb if index is None else index.shape[2]
    index = np.zeros((L, Hkv, Bcap, D), dtype=np.uint16) if index is None else np.array(index, dtype=np.uint16, copy=True)
    mean = np.zeros((L, Hkv, nb, D)) if return_mean else None
    sp = None if src_pos is None else _c(src_pos, np.int32)
    lib.orc_meank_build(_ptr(k), L, Hkv, T, D, block, first_block, _ptr(sp), float(rope_base),
                        int(rope_style), _ptr(index), Bcap, _ptr(mean))
    return (index, mean) if return_mean else index


def block_mass(q, index, n_blocks, n_sink, n_recent, l, g, Hkv=None):
    """Unnormalised candidate mass row of one (l, g); q bf16 [L,Hq,M,D], index [L,Hkv,Bcap,D]."""
    lib = _load()
    qq = _c(q, np.uint16)
    ix = _c(index, np.uint16)
    L, Hq, M, D = qq.shape
    Hkv = ix.shape[1]
    Bcap = ix.shape[2]
    part = np.zeros(n_blocks)
    lib.orc_block_mass(_ptr(qq), _ptr(ix), L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent,
                       int(l), int(g), _ptr(part))
    return part


def block_scores(q, index, n_blocks, n_sink, n_recent, return_partial=False):
    """R_b over n_blocks; q bf16 bits [L,Hq,M,D], index bf16 bits [L,Hkv,Bcap,D]."""
    lib = _load()
    qq = _c(q, np.uint16)
    ix = _c(index, np.uint16)
    L, Hq, M, D = qq.shape
    Hkv, Bcap = ix.shape[1], ix.shape[2]
    R = np.zeros(n_blocks)
    part = np.zeros((L * Hkv, n_blocks)) if return_partial else None
    lib.orc_block_scores(_ptr(qq), _ptr(ix), L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent,
                         _ptr(R), _ptr(part))
    return (R, part) if return_partial else R


def select_blocks(R, n_sink, n_recent, k):
    lib = _load()
    r = _c(R, np.float64)
    ids = np.zeros(max(r.size, 1), dtype=np.int32)
    n = lib.orc_select_blocks(_ptr(r), r.size, n_sink, n_recent, k, _ptr(ids))
    return ids[:n].copy()


def rerope_scatter(k_src, src_block, dst_page, dst_pos0, pool, page, rope_base,
                   rope_style=ROPE_NEOX, src_layer_stride=None, src_head_stride=None, L=None, Hkv=None):
    """Returns a new pool (bf16 bits [L,P,page,Hkv,D]) with the scattered, re-rotated rows."""
    lib = _load()
    k = _c(k_src, np.uint16)
    out = np.array(pool, dtype=np.uint16, copy=True)
    Lp, P, pg, Hk, D = out.shape
    assert pg == page
    L = Lp if L is None else L
    Hkv = Hk if Hkv is None else Hkv
    if src_head_stride is None:
        src_head_stride = k.shape[-2] * D
    if src_layer_stride is None:
        src_layer_stride = Hkv * src_head_stride
    sb = _c(src_block, np.int32)
    dp = _c(dst_page, np.int32)
    d0 = _c(dst_pos0, np.int32)
    lib.orc_rerope_scatter(_ptr(k), int(src_layer_stride), int(src_head_stride), _ptr(sb), _ptr(dp),
                           _ptr(d0), sb.size, L, Hkv, D, page, float(rope_base), int(rope_style),
                           _ptr(out), P)
    return out


def workset_diff(prev_ids, prev_pages, new_ids, P, page):
    """Differential working-set update (KVMEM restore path).

    Returns a dict with new_pages, shift [n_new]; in_rank, in_page (incoming);
    mv_rank, mv_shift (retained blocks whose position moved); out_page
    (released pages).  Raises ValueError when the pool has too few free pages."""
    lib = _load()
    pi = _c(prev_ids, np.int32)
    pp = _c(prev_pages, np.int32)
    ni = _c(new_ids, np.int32)
    n_prev, n_new = pi.size, ni.size
    new_pages = np.zeros(max(n_new, 1), np.int32)
    shift = np.zeros(max(n_new, 1), np.int32)
    in_rank = np.zeros(max(n_new, 1), np.int32)
    in_page = np.zeros(max(n_new, 1), np.int32)
    mv_rank = np.zeros(max(n_new, 1), np.int32)
    mv_shift = np.zeros(max(n_new, 1), np.int32)
    out_page = np.zeros(max(n_prev, 1), np.int32)
    counts = np.zeros(3, np.int32)
    rc = lib.orc_workset_diff(_ptr(pi), _ptr(pp), n_prev, _ptr(ni), n_new, int(P), int(page), _ptr(new_pages),
                              _ptr(shift), _ptr(in_rank), _ptr(in_page), _ptr(mv_rank), _ptr(mv_shift),
                              _ptr(out_page), _ptr(counts))
    if rc != 0:
        raise ValueError("workset_diff: not enough free pages")
    n_in, n_mv, n_out = (int(c) for c in counts)
    return {"new_pages": new_pages[:n_new].copy(), "shift": shift[:n_new].copy(),
            "in_rank": in_rank[:n_in].copy(), "in_page": in_page[:n_in].copy(),
            "mv_rank": mv_rank[:n_mv].copy(), "mv_shift": mv_shift[:n_mv].copy(),
            "out_page": out_page[:n_out].copy()}


def restore_blocks(k_src, v_src, src_block, dst_page, dst_pos0, k_pool, v_pool, page, rope_base,
                   rope_style=ROPE_NEOX):
    """Incoming-block restore: K re-rotated to its compact position, V copied.

    k_src, v_src: bf16 bits [L,Hkv,T,D]; pools bf16 bits [L,P,page,Hkv,D].
    Returns new (k_pool, v_pool)."""
    lib = _load()
    k = _c(k_src, np.uint16)
    v = _c(v_src, np.uint16)
    assert k.shape == v.shape
    ko = np.array(k_pool, dtype=np.uint16, copy=True)
    vo = np.array(v_pool, dtype=np.uint16, copy=True)
    L, Hkv, T, D = k.shape
    P = ko.shape[1]
    sb = _c(src_block, np.int32)
    dp = _c(dst_page, np.int32)
    d0 = _c(dst_pos0, np.int32)
    lib.orc_restore_blocks(_ptr(k), _ptr(v), Hkv * T * D, T * D, _ptr(sb), _ptr(dp), _ptr(d0), sb.size, L, Hkv, D,
                           page, float(rope_base), int(rope_style), _ptr(ko), _ptr(vo), P)
    return ko, vo


def rerope_shift(pool, pages, shifts, page, rope_base, rope_style=ROPE_NEOX):
    """Turn every row of the listed pages by shifts[i] positions; returns a new pool."""
    lib = _load()
    out = np.array(pool, dtype=np.uint16, copy=True)
    L, P, pg, Hkv, D = out.shape
    assert pg == page
    pg_ = _c(pages, np.int32)
    sh = _c(shifts, np.int32)
    lib.orc_rerope_shift(_ptr(out), P, _ptr(pg_), _ptr(sh), pg_.size, L, Hkv, D, page, float(rope_base),
                         int(rope_style))
    return out


def span_keep(span_start, span_end, del_ids, N, keep_in=None):
    """SideQuest cursor eviction: keep mask with the listed cursors' spans cleared.

    Returns (keep_out uint8 [N], number of ids outside the cursor table)."""
    lib = _load()
    ss, se = _c(span_start, np.int32), _c(span_end, np.int32)
    di = _c(del_ids, np.int32)
    ki = None if keep_in is None else _c(keep_in, np.uint8)
    out = np.zeros(max(N, 1), np.uint8)
    bad = lib.orc_span_keep(_ptr(ss), _ptr(se), ss.size, _ptr(di), di.size, _ptr(ki), int(N), _ptr(out))
    return out[:N].copy(), int(bad)


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (OCP 8-bit float: bias 7, 3 mantissa bits, max 448)."""
    return float(_load().orc_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(y: float) -> int:
    """Nearest E4M3 code to y (|y| <= 448), ties to the even code; the sign of zero is kept."""
    return int(_load().orc_e4m3_encode(float(y)))


def fp8_row_exp(x) -> int:
    """Scale exponent of an index row: the smallest e >= -100 with max|x| <= 448 * 2^e."""
    v = _c(x, np.float64)
    return int(_load().orc_fp8_row_exp(_ptr(v), v.size))


def index_to_fp8(index_bits):
    """Mean-K index rows [..., D] (bf16 bits) -> (E4M3 codes uint8 [..., D], scale exponents int8 [...]).
    Each row is stored as its codes and 2^e: value = code * 2^e."""
    b = _c(index_bits, np.uint16)
    D = b.shape[-1]
    rows = b.size // D
    codes = np.empty(b.shape, dtype=np.uint8)
    exps = np.empty(b.shape[:-1], dtype=np.int8)
    _load().orc_index_to_fp8(_ptr(b), rows, D, _ptr(codes), _ptr(exps))
    return codes, exps


def index_from_fp8(codes, exps):
    """E4M3 codes [..., D] and scale exponents [...] -> bf16 bits [..., D] (every value is exact in bf16)."""
    c = _c(codes, np.uint8)
    e = _c(exps, np.int8)
    D = c.shape[-1]
    rows = c.size // D
    assert e.size == rows
    out = np.empty(c.shape, dtype=np.uint16)
    _load().orc_index_from_fp8(_ptr(c), _ptr(e), rows, D, _ptr(out))
    return out
