"""kv_cache_retention_gb300: Python binding of libkvsel, the GB300 library for
query-driven KV-cache retention scoring and selection (IntentKV rule scoring
with dead-slot redirect; KVMEM Mean-K block retrieval with re-RoPE restore).

The binding only marshals arguments: every step runs in the CUDA kernels of
``libkvsel.so`` (built in-tree by ``_build.build()``).  Importing this package
fails loudly when the library is missing; there is no fallback.

Two layers:
  * module functions ``kvsel_*`` with exactly the C signatures (raw pointers
    as ints, sizes, stream handle) from ``include/kvsel.h``;
  * ``Context``: the same calls taking torch tensors, checking dtype, device
    and contiguity, and passing ``data_ptr()`` plus the current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvsel.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_SHAPE = -2
ERR_ALIGN = -3
ERR_UNSUPPORTED = -4
ERR_CUDA = -5
ERR_TIMEOUT = -6
ERR_DEVICE_CHECK = -7

F32 = 0
BF16 = 1
ROPE_NEOX = 0
ROPE_INTERLEAVED = 1
STAGE_AUTO = 0    # kvsel_stage_restore: direct when the repository is pinned, else packed
STAGE_PACKED = 1  # gather into pinned batches, copy, restore (pipelined)
STAGE_DIRECT = 2  # the restore kernel reads the pinned repository in place

# name -> (restype, argtypes), mirroring include/kvsel.h
_P, _I, _I64, _F, _D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
_IP = ctypes.POINTER(ctypes.c_int)
class MemorySession(ctypes.Structure):
    """kvsel_memory_session (include/kvsel.h)."""
    _fields_ = [("q_rows", ctypes.c_void_p), ("R", ctypes.c_int), ("lam", ctypes.c_float),
                ("first_turn", ctypes.c_int), ("M", ctypes.c_void_p), ("A", ctypes.c_void_p)]


class RuleSession(ctypes.Structure):
    """kvsel_rule_session (include/kvsel.h)."""
    _fields_ = [("slot_map", ctypes.c_void_p), ("N", ctypes.c_int), ("M", ctypes.c_void_p), ("pi", ctypes.c_int),
                ("q_s", ctypes.c_int), ("q_e", ctypes.c_int), ("rule", ctypes.c_void_p)]


class TopkSession(ctypes.Structure):
    """kvsel_topk_session (include/kvsel.h)."""
    _fields_ = [("rule", ctypes.c_void_p), ("N", ctypes.c_int), ("pi", ctypes.c_int), ("q_s", ctypes.c_int),
                ("q_e", ctypes.c_int), ("C", ctypes.c_int), ("keep", ctypes.c_void_p), ("keep_idx", ctypes.c_void_p)]


SIGNATURES = {
    "kvsel_version": (_I, []),
    "kvsel_ctx_create": (_I, [_I, ctypes.POINTER(_P)]),
    "kvsel_ctx_destroy": (_I, [_P]),
    "kvsel_last_error_string": (ctypes.c_char_p, [_P]),
    "kvsel_check_device": (_I, [_P, _P]),
    "kvsel_memory_update": (_I, [_P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P]),
    "kvsel_rule_scores": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I64, _I64, _P, _I, _I, _I, _P, _P]),
    "kvsel_rule_scores_noalloc": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I64, _I64, _P, _I, _I, _I, _P, _P]),
    "kvsel_topk_retain": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _IP, _P]),
    "kvsel_redirect_slots": (_I, [_P, _P, _P, _I, ctypes.c_int32, _P, _P]),
    "kvsel_meank_build": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _D, _I, _P, _I, _P]),
    "kvsel_block_scores": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "kvsel_select_blocks": (_I, [_P, _P, _I, _I, _I, _I, _P, _IP, _P]),
    "kvsel_rerope_scatter": (_I, [_P, _P, _I64, _I64, _I, _P, _P, _P, _I, _I, _I, _I, _I, _D, _I, _P, _I, _P]),
    "kvsel_memory_update_batch": (_I, [_P, _I, _I, _I, _I, _I, _P, _I, _P]),
    "kvsel_rule_scores_batch": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I64, _I64, _P, _I, _P]),
    "kvsel_topk_retain_batch": (_I, [_P, _P, _I, _P, _P]),
    "kvsel_span_keep": (_I, [_P, _P, _P, _I, _P, _I, _P, _I, _P, _P]),
    "kvsel_index_to_fp8": (_I, [_P, _P, _I64, _I, _P, _P, _P]),
    "kvsel_index_from_fp8": (_I, [_P, _P, _P, _I64, _I, _P, _P]),
    "kvsel_workset_diff": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "kvsel_restore_blocks": (_I, [_P, _P, _P, _I64, _I64, _I, _P, _P, _P, _I, _P, _I, _I, _I, _I, _D, _I, _P, _P,
                                  _I, _P]),
    "kvsel_rerope_shift": (_I, [_P, _P, _I, _P, _P, _I, _P, _I, _I, _I, _I, _D, _I, _P]),
    "kvsel_stage_restore": (_I, [_P, _P, _P, _I64, _I64, _I, _P, _P, _P, _I, _I, _I, _I, _I, _D, _I, _P, _P, _I,
                                 _I, _I, _I, _P]),
}


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"libkvsel.so not found at {_LIB_PATH}: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
LIB_PATH = _LIB_PATH


class KvselError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"kvsel error {code}: {msg}")
        self.code = code


# ---------------------------------------------------------------------------
# raw C-ABI functions (same names and argument order as include/kvsel.h)
# ---------------------------------------------------------------------------

def kvsel_version() -> int:
    return _lib.kvsel_version()


def kvsel_ctx_create(device: int) -> int:
    h = _P()
    rc = _lib.kvsel_ctx_create(device, ctypes.byref(h))
    if rc != OK:
        raise KvselError(rc, f"kvsel_ctx_create(device={device}) failed")
    return h.value


def kvsel_ctx_destroy(ctx: int) -> int:
    return _lib.kvsel_ctx_destroy(ctx)


def kvsel_last_error_string(ctx: int) -> str:
    return _lib.kvsel_last_error_string(ctx).decode()


def kvsel_check_device(ctx, stream):
    return _lib.kvsel_check_device(ctx, stream)


def kvsel_memory_update(ctx, q_rows, q_dtype, L, Hq, R, D, lam, first_turn, norm_mode, M, A, stream):
    return _lib.kvsel_memory_update(ctx, q_rows, q_dtype, L, Hq, R, D, lam, first_turn, norm_mode, M, A, stream)


def kvsel_rule_scores(ctx, k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N, D, layer_stride, slot_stride, M,
                      pi, q_s, q_e, rule, stream):
    return _lib.kvsel_rule_scores(ctx, k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N, D, layer_stride,
                                  slot_stride, M, pi, q_s, q_e, rule, stream)


def kvsel_rule_scores_noalloc(ctx, k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N, D, layer_stride, slot_stride,
                              M, pi, q_s, q_e, rule, stream):
    """kvsel_rule_scores on the library's fixed scratch array: no device allocation
    (for callers that cannot allocate; sizes needing more than 64 MiB of scratch
    are rejected)."""
    return _lib.kvsel_rule_scores_noalloc(ctx, k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N, D, layer_stride,
                                          slot_stride, M, pi, q_s, q_e, rule, stream)


def kvsel_topk_retain(ctx, score, N, pi, q_s, q_e, C, keep, keep_idx, n_keep_host, stream):
    return _lib.kvsel_topk_retain(ctx, score, N, pi, q_s, q_e, C, keep, keep_idx, n_keep_host, stream)


def kvsel_redirect_slots(ctx, slot_in, keep, N, dead_slot, slot_out, stream):
    return _lib.kvsel_redirect_slots(ctx, slot_in, keep, N, dead_slot, slot_out, stream)


def kvsel_meank_build(ctx, k_src, L, Hkv, T, D, block, first_block, src_pos, rope_base, rope_style, index, Bcap,
                      stream):
    return _lib.kvsel_meank_build(ctx, k_src, L, Hkv, T, D, block, first_block, src_pos, rope_base, rope_style,
                                  index, Bcap, stream)


def kvsel_block_scores(ctx, q, index, L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent, R, R_partial, stream):
    return _lib.kvsel_block_scores(ctx, q, index, L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent, R, R_partial,
                                   stream)


def kvsel_select_blocks(ctx, R, n_blocks, n_sink, n_recent, k, ids, n_sel_host, stream):
    return _lib.kvsel_select_blocks(ctx, R, n_blocks, n_sink, n_recent, k, ids, n_sel_host, stream)


def kvsel_rerope_scatter(ctx, k_src, src_layer_stride, src_head_stride, src_tokens, src_block, dst_page, dst_pos0,
                         n, L, Hkv, D, page, rope_base, rope_style, pool, P, stream):
    return _lib.kvsel_rerope_scatter(ctx, k_src, src_layer_stride, src_head_stride, src_tokens, src_block, dst_page,
                                     dst_pos0, n, L, Hkv, D, page, rope_base, rope_style, pool, P, stream)


def kvsel_memory_update_batch(ctx, q_dtype, L, Hq, D, norm_mode, sessions, S, stream):
    return _lib.kvsel_memory_update_batch(ctx, q_dtype, L, Hq, D, norm_mode, sessions, S, stream)


def kvsel_rule_scores_batch(ctx, k_pool, k_dtype, n_slots, L, Hq, Hkv, D, layer_stride, slot_stride, sessions, S,
                            stream):
    return _lib.kvsel_rule_scores_batch(ctx, k_pool, k_dtype, n_slots, L, Hq, Hkv, D, layer_stride, slot_stride,
                                        sessions, S, stream)


def kvsel_topk_retain_batch(ctx, sessions, S, n_keep_host, stream):
    return _lib.kvsel_topk_retain_batch(ctx, sessions, S, n_keep_host, stream)


def kvsel_span_keep(ctx, span_start, span_end, n_cursors, del_ids, n_del, keep_in, N, keep_out, stream):
    return _lib.kvsel_span_keep(ctx, span_start, span_end, n_cursors, del_ids, n_del, keep_in, N, keep_out, stream)


def kvsel_index_to_fp8(ctx, index, rows, D, codes, exps, stream):
    return _lib.kvsel_index_to_fp8(ctx, index, rows, D, codes, exps, stream)


def kvsel_index_from_fp8(ctx, codes, exps, rows, D, index, stream):
    return _lib.kvsel_index_from_fp8(ctx, codes, exps, rows, D, index, stream)


def kvsel_workset_diff(ctx, prev_ids, prev_pages, n_prev, new_ids, n_new, P, page, new_pages, shift, in_rank,
                       in_page, mv_rank, mv_shift, out_page, counts, stream):
    return _lib.kvsel_workset_diff(ctx, prev_ids, prev_pages, n_prev, new_ids, n_new, P, page, new_pages, shift,
                                   in_rank, in_page, mv_rank, mv_shift, out_page, counts, stream)


def kvsel_restore_blocks(ctx, k_src, v_src, src_layer_stride, src_head_stride, src_tokens, src_block, dst_page,
                         dst_pos0, n, n_dev, L, Hkv, D, page, rope_base, rope_style, k_pool, v_pool, P, stream):
    return _lib.kvsel_restore_blocks(ctx, k_src, v_src, src_layer_stride, src_head_stride, src_tokens, src_block,
                                     dst_page, dst_pos0, n, n_dev, L, Hkv, D, page, rope_base, rope_style, k_pool,
                                     v_pool, P, stream)


def kvsel_rerope_shift(ctx, pool, P, pages, shifts, n, n_dev, L, Hkv, D, page, rope_base, rope_style, stream):
    return _lib.kvsel_rerope_shift(ctx, pool, P, pages, shifts, n, n_dev, L, Hkv, D, page, rope_base, rope_style,
                                   stream)


def kvsel_stage_restore(ctx, host_k, host_v, host_layer_stride, host_head_stride, host_tokens, blocks, dst_page,
                        dst_pos0, n, L, Hkv, D, page, rope_base, rope_style, k_pool, v_pool, P, chunk_blocks,
                        gather_threads, mode, stream):
    return _lib.kvsel_stage_restore(ctx, host_k, host_v, host_layer_stride, host_head_stride, host_tokens, blocks,
                                    dst_page, dst_pos0, n, L, Hkv, D, page, rope_base, rope_style, k_pool, v_pool,
                                    P, chunk_blocks, gather_threads, mode, stream)


# ---------------------------------------------------------------------------
# tensor-level wrapper
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t, dtype=None, name="tensor"):
    """data_ptr of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (libkvsel has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


_raw_stream_getter = None


def _current_stream(device):
    """Handle of the current CUDA stream of `device`.  torch's raw getter returns it
    directly (about 0.2 us, against about 3 us for the Stream object), which matters for
    the µs-scale calls; the public API is the fallback."""
    global _raw_stream_getter
    if _raw_stream_getter is None:
        torch = _torch()
        f = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _raw_stream_getter = f if f is not None else (lambda d: torch.cuda.current_stream(d).cuda_stream)
    return _raw_stream_getter(device)


def _code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


class Context:
    """A libkvsel context on one CUDA device; methods mirror the C calls."""

    def __init__(self, device: int = 0):
        self.device = device
        self.handle = kvsel_ctx_create(device)

    def close(self):
        if self.handle:
            kvsel_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _stream(self, stream):
        if stream is not None:
            return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        return _current_stream(self.device)

    def _check(self, rc):
        if rc != OK:
            raise KvselError(rc, kvsel_last_error_string(self.handle))

    def check_device(self, stream=None):
        self._check(kvsel_check_device(self.handle, self._stream(stream)))

    # IntentKV -------------------------------------------------------------
    def memory_update(self, q_rows, lam, M, first_turn=False, norm_mode=0, A=None, stream=None):
        torch = _torch()
        L, Hq, R, D = q_rows.shape
        self._check(kvsel_memory_update(self.handle, _ptr(q_rows, name="q_rows"), _code(q_rows), L, Hq, R, D,
                                        float(lam), int(bool(first_turn)), int(norm_mode),
                                        _ptr(M, torch.float32, "M"), _ptr(A, torch.float32, "A"),
                                        self._stream(stream)))

    def rule_scores(self, k_pool, M, L, Hq, Hkv, N, D, pi, q_s, q_e, rule, slot_map=None, n_slots=None,
                    layer_stride=None, slot_stride=None, stream=None):
        torch = _torch()
        if slot_stride is None:
            slot_stride = Hkv * D
        if n_slots is None:
            n_slots = k_pool.numel() // (L * slot_stride)
        if layer_stride is None:
            layer_stride = n_slots * slot_stride
        self._check(kvsel_rule_scores(self.handle, _ptr(k_pool, name="k_pool"), _code(k_pool),
                                      _ptr(slot_map, torch.int32, "slot_map"), int(n_slots), L, Hq, Hkv, N, D,
                                      int(layer_stride), int(slot_stride), _ptr(M, torch.float32, "M"),
                                      pi, q_s, q_e, _ptr(rule, torch.float32, "rule"), self._stream(stream)))

    def topk_retain(self, score, pi, q_s, q_e, C, keep=None, keep_idx=None, stream=None):
        torch = _torch()
        n = ctypes.c_int(0)
        self._check(kvsel_topk_retain(self.handle, _ptr(score, torch.float32, "score"), score.numel(), pi, q_s,
                                      q_e, C, _ptr(keep, torch.uint8, "keep"), _ptr(keep_idx, torch.int32, "keep_idx"),
                                      ctypes.byref(n), self._stream(stream)))
        return n.value

    def redirect_slots(self, slot_in, keep, dead_slot, slot_out, stream=None):
        torch = _torch()
        self._check(kvsel_redirect_slots(self.handle, _ptr(slot_in, torch.int32, "slot_in"),
                                         _ptr(keep, torch.uint8, "keep"), slot_in.numel(), int(dead_slot),
                                         _ptr(slot_out, torch.int32, "slot_out"), self._stream(stream)))

    # KVMEM ----------------------------------------------------------------
    def meank_build(self, k_src, block, index, first_block=0, src_pos=None, rope_base=1e6, rope_style=ROPE_NEOX,
                    stream=None):
        torch = _torch()
        L, Hkv, T, D = k_src.shape
        self._check(kvsel_meank_build(self.handle, _ptr(k_src, torch.bfloat16, "k_src"), L, Hkv, T, D, block,
                                      first_block, _ptr(src_pos, torch.int32, "src_pos"), float(rope_base),
                                      int(rope_style), _ptr(index, torch.bfloat16, "index"), index.shape[2],
                                      self._stream(stream)))

    def block_scores(self, q, index, n_blocks, n_sink, n_recent, R, R_partial=None, stream=None):
        torch = _torch()
        L, Hq, M, D = q.shape
        Hkv, Bcap = index.shape[1], index.shape[2]
        self._check(kvsel_block_scores(self.handle, _ptr(q, torch.bfloat16, "q"), _ptr(index, torch.bfloat16, "index"),
                                       L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent,
                                       _ptr(R, torch.float32, "R"), _ptr(R_partial, torch.float32, "R_partial"),
                                       self._stream(stream)))

    def select_blocks(self, R, n_sink, n_recent, k, ids, n_blocks=None, stream=None):
        torch = _torch()
        n = ctypes.c_int(0)
        nb = R.numel() if n_blocks is None else n_blocks
        self._check(kvsel_select_blocks(self.handle, _ptr(R, torch.float32, "R"), nb, n_sink, n_recent, k,
                                        _ptr(ids, torch.int32, "ids"), ctypes.byref(n), self._stream(stream)))
        return n.value

    def rerope_scatter(self, k_src, src_block, dst_page, dst_pos0, pool, rope_base, rope_style=ROPE_NEOX,
                       n=None, stream=None):
        """k_src: bf16 [L][Hkv][T][D] (contiguous); pool: bf16 [L][P][page][Hkv][D]."""
        torch = _torch()
        L, Hkv, T, D = k_src.shape
        _, P, page, _, _ = pool.shape
        n = src_block.numel() if n is None else n
        self._check(kvsel_rerope_scatter(self.handle, _ptr(k_src, torch.bfloat16, "k_src"), Hkv * T * D, T * D, T,
                                         _ptr(src_block, torch.int32, "src_block"),
                                         _ptr(dst_page, torch.int32, "dst_page"),
                                         _ptr(dst_pos0, torch.int32, "dst_pos0"), n, L, Hkv, D, page,
                                         float(rope_base), int(rope_style), _ptr(pool, torch.bfloat16, "pool"), P,
                                         self._stream(stream)))

    # batched sessions ------------------------------------------------------

    def memory_update_batch(self, q_rows_list, lam_list, M_list, first_turn_list=None, norm_mode=0, A_list=None,
                            stream=None):
        """One QueryMemory turn for each session: q_rows_list[i] [L][Hq][R_i][D] (same dtype for all)."""
        torch = _torch()
        S = len(q_rows_list)
        if S == 0:
            return
        q0 = q_rows_list[0]
        L, Hq, _, D = q0.shape
        dt = BF16 if q0.dtype == torch.bfloat16 else F32
        arr = (MemorySession * S)()
        for i, q in enumerate(q_rows_list):
            if q.dtype != q0.dtype or tuple(q.shape[:2]) != (L, Hq) or q.shape[3] != D:
                raise ValueError("memory_update_batch: sessions must share dtype, L, Hq and D")
            ft = bool(first_turn_list[i]) if first_turn_list is not None else False
            A = None if A_list is None else A_list[i]
            arr[i] = MemorySession(_ptr(q, name="q_rows"), q.shape[2], float(lam_list[i]), int(ft),
                                   _ptr(M_list[i], torch.float32, "M"), _ptr(A, torch.float32, "A"))
        self._check(kvsel_memory_update_batch(self.handle, dt, L, Hq, D, int(norm_mode), arr, S, self._stream(stream)))

    def rule_scores_batch(self, k_pool, M_list, L, Hq, Hkv, N_list, D, forced_list, rule_list, slot_maps=None,
                          n_slots=None, layer_stride=None, slot_stride=None, stream=None):
        """rule_scores for many sessions on one shared pool; forced_list[i] = (pi, q_s, q_e)."""
        torch = _torch()
        S = len(M_list)
        dt = BF16 if k_pool.dtype == torch.bfloat16 else F32
        if slot_stride is None:
            slot_stride = Hkv * D
        if n_slots is None:
            n_slots = k_pool.numel() // (L * slot_stride)
        if layer_stride is None:
            layer_stride = n_slots * slot_stride
        arr = (RuleSession * S)()
        for i in range(S):
            sm = None if slot_maps is None else slot_maps[i]
            pi, qs, qe = forced_list[i]
            arr[i] = RuleSession(_ptr(sm, torch.int32, "slot_map"), int(N_list[i]), _ptr(M_list[i], torch.float32, "M"),
                                 int(pi), int(qs), int(qe), _ptr(rule_list[i], torch.float32, "rule"))
        self._check(kvsel_rule_scores_batch(self.handle, _ptr(k_pool, None, "k_pool"), dt, int(n_slots), L, Hq, Hkv, D,
                                            int(layer_stride), int(slot_stride), arr, S, self._stream(stream)))

    def topk_retain_batch(self, rule_list, forced_list, C_list, keep_list=None, keep_idx_list=None, stream=None):
        """topk_retain for many sessions; returns the host list of |keep| per session."""
        torch = _torch()
        S = len(rule_list)
        arr = (TopkSession * S)()
        for i, r in enumerate(rule_list):
            pi, qs, qe = forced_list[i]
            keep = None if keep_list is None else keep_list[i]
            idx = None if keep_idx_list is None else keep_idx_list[i]
            arr[i] = TopkSession(_ptr(r, torch.float32, "rule"), r.numel(), int(pi), int(qs), int(qe), int(C_list[i]),
                                 _ptr(keep, torch.uint8, "keep"), _ptr(idx, torch.int32, "keep_idx"))
        n_keep = (ctypes.c_int * max(S, 1))()
        self._check(kvsel_topk_retain_batch(self.handle, arr, S, n_keep, self._stream(stream)))
        return [int(n_keep[i]) for i in range(S)]

    def span_keep(self, span_start, span_end, del_ids, N, keep_out, keep_in=None, stream=None):
        """Clear the listed cursors' spans from a keep mask (uint8 CUDA tensors; keep_out may be keep_in)."""
        torch = _torch()
        n_cur, n_del = span_start.numel(), del_ids.numel()
        i32 = torch.int32
        self._check(kvsel_span_keep(self.handle, _ptr(span_start, i32, "span_start") if n_cur else None,
                                    _ptr(span_end, i32, "span_end") if n_cur else None, n_cur,
                                    _ptr(del_ids, i32, "del_ids") if n_del else None, n_del,
                                    _ptr(keep_in, torch.uint8, "keep_in"), int(N),
                                    _ptr(keep_out, torch.uint8, "keep_out"), self._stream(stream)))

    def index_to_fp8(self, index, codes=None, exps=None, stream=None):
        """bf16 index [..., D] -> (E4M3 codes uint8 [..., D], scale exponents int8 [...]) as CUDA tensors."""
        torch = _torch()
        D = index.shape[-1]
        rows = index.numel() // D if D else 0
        if codes is None:
            codes = torch.empty(index.shape, dtype=torch.uint8, device=index.device)
        if exps is None:
            exps = torch.empty(index.shape[:-1], dtype=torch.int8, device=index.device)
        self._check(kvsel_index_to_fp8(self.handle, _ptr(index, torch.bfloat16, "index"), rows, D,
                                       _ptr(codes, torch.uint8, "codes"), _ptr(exps, torch.int8, "exps"),
                                       self._stream(stream)))
        return codes, exps

    def index_from_fp8(self, codes, exps, index=None, stream=None):
        """E4M3 codes [..., D] and exponents [...] -> bf16 index [..., D] (CUDA tensors)."""
        torch = _torch()
        D = codes.shape[-1]
        rows = codes.numel() // D if D else 0
        if index is None:
            index = torch.empty(codes.shape, dtype=torch.bfloat16, device=codes.device)
        self._check(kvsel_index_from_fp8(self.handle, _ptr(codes, torch.uint8, "codes"), _ptr(exps, torch.int8, "exps"),
                                         rows, D, _ptr(index, torch.bfloat16, "index"), self._stream(stream)))
        return index

    def workset_diff(self, prev_ids, prev_pages, new_ids, P, page, out=None, stream=None):
        """Retained / incoming / outgoing split of a new working set (int32 CUDA tensors).

        Returns a dict of device tensors: new_pages, shift, in_rank, in_page,
        mv_rank, mv_shift (length n_new, valid prefixes given by counts), out_page
        (length n_prev) and counts = (n_incoming, n_moved, n_outgoing).  Nothing
        is synchronised; read counts on the host only when the sizes are needed."""
        torch = _torch()
        n_prev, n_new = prev_ids.numel(), new_ids.numel()
        dev = new_ids.device if n_new else prev_ids.device
        if out is None:
            out = {k: torch.empty(max(n_new, 1), dtype=torch.int32, device=dev)
                   for k in ("new_pages", "shift", "in_rank", "in_page", "mv_rank", "mv_shift")}
            out["out_page"] = torch.empty(max(n_prev, 1), dtype=torch.int32, device=dev)
            out["counts"] = torch.zeros(3, dtype=torch.int32, device=dev)
        i32 = torch.int32
        self._check(kvsel_workset_diff(
            self.handle, _ptr(prev_ids, i32, "prev_ids") if n_prev else None,
            _ptr(prev_pages, i32, "prev_pages") if n_prev else None, n_prev,
            _ptr(new_ids, i32, "new_ids") if n_new else None, n_new, int(P), int(page),
            _ptr(out["new_pages"], i32), _ptr(out["shift"], i32), _ptr(out["in_rank"], i32),
            _ptr(out["in_page"], i32), _ptr(out["mv_rank"], i32), _ptr(out["mv_shift"], i32),
            _ptr(out["out_page"], i32), _ptr(out["counts"], i32), self._stream(stream)))
        return out

    def restore_blocks(self, k_src, v_src, src_block, dst_page, dst_pos0, k_pool, v_pool, rope_base,
                       rope_style=ROPE_NEOX, n=None, n_dev=None, stream=None):
        """k_src, v_src: bf16 [L][Hkv][T][D] (contiguous, same shape); pools bf16 [L][P][page][Hkv][D]."""
        torch = _torch()
        L, Hkv, T, D = k_src.shape
        if tuple(v_src.shape) != tuple(k_src.shape) or tuple(v_pool.shape) != tuple(k_pool.shape):
            raise ValueError("restore_blocks: V source and pool must match K's shapes")
        _, P, page, _, _ = k_pool.shape
        n = src_block.numel() if n is None else n
        bf = torch.bfloat16
        self._check(kvsel_restore_blocks(self.handle, _ptr(k_src, bf, "k_src"), _ptr(v_src, bf, "v_src"), Hkv * T * D,
                                         T * D, T, _ptr(src_block, torch.int32, "src_block"),
                                         _ptr(dst_page, torch.int32, "dst_page"),
                                         _ptr(dst_pos0, torch.int32, "dst_pos0"), n,
                                         _ptr(n_dev, torch.int32, "n_dev"), L, Hkv, D, page, float(rope_base),
                                         int(rope_style), _ptr(k_pool, bf, "k_pool"), _ptr(v_pool, bf, "v_pool"), P,
                                         self._stream(stream)))

    def stage_restore(self, host_k, host_v, blocks, dst_page, dst_pos0, k_pool, v_pool, rope_base,
                      rope_style=ROPE_NEOX, chunk_blocks=64, gather_threads=None, mode=None, stream=None):
        """Restore blocks from a host repository (CPU bf16 tensors [L][Hkv][T][D], pinned or not) into the
        device pools, through the packed, pipelined host -> device staging.  blocks, dst_page and dst_pos0
        are host int32 arrays (numpy or CPU tensors)."""
        import numpy as np
        torch = _torch()
        for name, t in (("host_k", host_k), ("host_v", host_v)):
            if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
                raise ValueError(f"{name}: expected a contiguous CPU bf16 tensor")
        if tuple(host_v.shape) != tuple(host_k.shape) or tuple(v_pool.shape) != tuple(k_pool.shape):
            raise ValueError("stage_restore: V repository and pool must match K's shapes")
        L, Hkv, T, D = host_k.shape
        _, P, page, _, _ = k_pool.shape
        arrs = [np.ascontiguousarray(np.asarray(a.cpu() if hasattr(a, "cpu") else a, dtype=np.int32))
                for a in (blocks, dst_page, dst_pos0)]
        n = arrs[0].size
        if any(a.size != n for a in arrs):
            raise ValueError("stage_restore: blocks, dst_page and dst_pos0 differ in length")
        ptrs = [a.ctypes.data_as(ctypes.c_void_p) for a in arrs]
        if gather_threads is None:
            gather_threads = min(16, os.cpu_count() or 1)
        self._check(kvsel_stage_restore(self.handle, ctypes.c_void_p(host_k.data_ptr()),
                                        ctypes.c_void_p(host_v.data_ptr()), Hkv * T * D, T * D, T, ptrs[0], ptrs[1],
                                        ptrs[2], n, L, Hkv, D, page, float(rope_base), int(rope_style),
                                        _ptr(k_pool, torch.bfloat16, "k_pool"), _ptr(v_pool, torch.bfloat16, "v_pool"),
                                        P, int(chunk_blocks), int(gather_threads),
                                        STAGE_AUTO if mode is None else int(mode), self._stream(stream)))

    def rerope_shift(self, pool, pages, shifts, rope_base, rope_style=ROPE_NEOX, n=None, n_dev=None, stream=None):
        """Turn the rows of the listed pages of pool (bf16 [L][P][page][Hkv][D]) by shifts[i] positions."""
        torch = _torch()
        L, P, page, Hkv, D = pool.shape
        n = pages.numel() if n is None else n
        self._check(kvsel_rerope_shift(self.handle, _ptr(pool, torch.bfloat16, "pool"), P,
                                       _ptr(pages, torch.int32, "pages"), _ptr(shifts, torch.int32, "shifts"), n,
                                       _ptr(n_dev, torch.int32, "n_dev"), L, Hkv, D, page, float(rope_base),
                                       int(rope_style), self._stream(stream)))
