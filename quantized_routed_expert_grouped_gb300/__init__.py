"""Grouped routed-expert decode for the verify window, GB300-native (sm_103a).

A thin ctypes binding over the C ABI in ``include/moe_grouped.h`` (library
``_build/libmoe_grouped.so``, built by ``build.py``). The functions here only marshal
arguments: torch tensors supply device memory and the current CUDA stream; every step runs in
the library's kernels. There is no CPU fallback: a missing library raises.

q8_1 rows are uint8 tensors of shape [rows, cols/32, 36].
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "Q8_0", "Q4B", "NL4", "CB2", "CB3", "CB3X", "CB2X", "MoeError", "transcode_cb", "lib", "row_bytes", "strerror",
    "quantize_q8_1", "route_group", "grouped_gu", "swiglu_q8_1", "grouped_down",
    "expert_grouped", "ExpertCall", "STATIC_SCRATCH_BYTES", "test_block_isum", "ERR_BITS", "F_PDL",
    "LayerCall", "layer_sync_ints", "router_topk", "combine", "F_SYNC_PAIR", "F_SYNC_ODD", "F_TEST_EXPIRE",
    "qsa_block_scores", "grouped_fused_sync_ints", "stage_blobs",
]

Q8_0, Q4B, NL4, CB2, CB3, CB3X, CB2X = 1, 2, 3, 4, 5, 6, 7
F_PDL = 1
F_SYNC_PAIR = 2  # moe_expert_layer: sync holds two halves used by alternate calls
F_SYNC_ODD = 4   # ... and this call uses the second half
F_TEST_EXPIRE = 8  # test hook: the down staging waits for a flag no call writes (timeout path)
STATIC_SCRATCH_BYTES = 4 << 20
ERR_BITS = {1: "NGROUPS", 2: "EXPERT", 4: "START", 8: "ENTRY", 16: "ALIGN", 32: "CODEBOOK",
            64: "TIMEOUT", 128: "ROUTE"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_grouped.so")
_LIB = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64


class MoeError(RuntimeError):
    pass


class WFmt(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int32), ("codebook", ctypes.c_void_p)]


class ExpertCallC(ctypes.Structure):
    _fields_ = [
        ("gu_fmt", WFmt), ("down_fmt", WFmt),
        ("n_embd", ctypes.c_int32), ("n_ff", ctypes.c_int32), ("n_experts", ctypes.c_int32),
        ("w_gu", _P), ("w_down", _P), ("grp_expert", _P), ("grp_start", _P), ("n_groups", _P),
        ("cap_groups", ctypes.c_int32), ("grid_groups", ctypes.c_int32), ("cap_entries", ctypes.c_int32),
        ("xq", _P), ("n_xq_rows", ctypes.c_int32), ("ent_src", _P), ("ent_dst", _P),
        ("gu", _P), ("hq", _P), ("out", _P), ("out_rows", ctypes.c_int64), ("out_row_stride", ctypes.c_int64),
        ("err", _P), ("flags", ctypes.c_int32),
    ]


class LayerCallC(ctypes.Structure):
    _fields_ = [
        ("gu_fmt", WFmt), ("down_fmt", WFmt),
        ("n_embd", ctypes.c_int32), ("n_ff", ctypes.c_int32), ("n_experts", ctypes.c_int32),
        ("w_gu", _P), ("w_down", _P), ("topk_ids", _P), ("T", ctypes.c_int32), ("k", ctypes.c_int32),
        ("x", _P), ("out", _P), ("out_row_stride", ctypes.c_int64), ("gu", _P), ("hq", _P), ("sync", _P),
        ("grp_expert", _P), ("grp_start", _P), ("n_groups", _P), ("ent_src", _P), ("ent_dst", _P), ("xq", _P),
        ("err", _P), ("flags", ctypes.c_int32),
    ]


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise MoeError(f"CUDA library not built: {LIB_PATH} (run __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        L.moe_row_bytes.argtypes = [_I, _I]
        L.moe_row_bytes.restype = _I64
        L.moe_strerror.argtypes = [_I]
        L.moe_strerror.restype = ctypes.c_char_p
        L.moe_quantize_q8_1.argtypes = [_P, _I64, _I64, _P, _P]
        L.moe_route_group.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]
        L.moe_grouped_gu.argtypes = [WFmt, _I, _I, _P, _I, _P, _P, _P, _I, _I, _P, _I, _P, _I, _P, _P, _P]
        L.moe_swiglu_q8_1.argtypes = [_P, _I, _P, _P, _I, _I, _P, _P, _P]
        L.moe_grouped_down.argtypes = [WFmt, _I, _I, _P, _I, _P, _P, _P, _I, _I, _P, _I, _P, _P, _I64, _I64,
                                       _P, _P]
        L.moe_expert_grouped.argtypes = [ctypes.POINTER(ExpertCallC), _P]
        L.moe_expert_grouped_static.argtypes = [ctypes.POINTER(ExpertCallC), _P]
        L.moe_test_block_isum.argtypes = [WFmt, _I, _P, _I, _P, _P, _P]
        L.moe_transcode_cb.argtypes = [WFmt, _I, _I, _I, _I, _P, _P, _P, _P]
        L.moe_expert_layer.argtypes = [ctypes.POINTER(LayerCallC), _P]
        L.moe_layer_sync_ints.argtypes = [_I, _I, _I]
        L.moe_layer_sync_ints.restype = _I64
        L.moe_router_topk.argtypes = [_P, _I, _I, _I, _P, _P, _P]
        L.moe_combine.argtypes = [_P, _I64, _P, _P, _I, _I, _I, _I, _P, _I64, _P]
        L.moe_qsa_block_scores.argtypes = [_P, _I, _P, _P, _I64, _P, _P]
        L.moe_expert_grouped_fused.argtypes = [ctypes.POINTER(ExpertCallC), _P, _P]
        L.moe_grouped_fused_sync_ints.argtypes = [_I, _I, _I]
        L.moe_grouped_fused_sync_ints.restype = _I64
        L.moe_stage_blobs.argtypes = [_P, _P, _P, _I, _P]
        for f in ("moe_quantize_q8_1", "moe_route_group", "moe_grouped_gu", "moe_swiglu_q8_1",
                  "moe_grouped_down", "moe_expert_grouped", "moe_expert_grouped_static", "moe_test_block_isum",
                  "moe_transcode_cb", "moe_expert_layer", "moe_router_topk", "moe_combine",
                  "moe_qsa_block_scores", "moe_expert_grouped_fused", "moe_stage_blobs"):
            getattr(L, f).restype = _I
        _LIB = L
    return _LIB


def row_bytes(typ: int, K: int) -> int:
    return int(lib().moe_row_bytes(typ, K))


def strerror(status: int) -> str:
    return lib().moe_strerror(status).decode()


def _check(rc: int):
    if rc != 0:
        raise MoeError(f"{rc}: {strerror(rc)}")


def _dp(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise MoeError("device tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _fmt(typ, codebook):
    return WFmt(typ, None if codebook is None else codebook.data_ptr())


def quantize_q8_1(x: torch.Tensor, xq: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """x: fp32 [rows, cols] (contiguous, device) -> uint8 q8_1 [rows, cols/32, 36]."""
    rows, cols = x.shape
    if xq is None:
        xq = torch.empty((rows, cols // 32, 36), dtype=torch.uint8, device=x.device)
    _check(lib().moe_quantize_q8_1(_dp(x), rows, cols, _dp(xq), _stream(stream)))
    return xq


def route_group(topk_ids, n_experts, entry_base, grp_expert, grp_start, n_groups, ent_src, ent_dst,
                err=None, stream=None):
    T, k = topk_ids.shape
    _check(lib().moe_route_group(_dp(topk_ids), T, k, n_experts, entry_base, _dp(grp_expert), _dp(grp_start),
                                 _dp(n_groups), _dp(ent_src), _dp(ent_dst), _dp(err), _stream(stream)))


def grouped_gu(typ, codebook, n_embd, n_ff, w_table, n_experts, grp_expert, grp_start, n_groups, cap_groups,
               grid_groups, xq, ent_src, cap_entries, gu, err=None, stream=None):
    _check(lib().moe_grouped_gu(_fmt(typ, codebook), n_embd, n_ff, _dp(w_table), n_experts, _dp(grp_expert),
                                _dp(grp_start), _dp(n_groups), cap_groups, grid_groups, _dp(xq), xq.shape[0],
                                _dp(ent_src), cap_entries, _dp(gu), _dp(err), _stream(stream)))


def swiglu_q8_1(gu, n_ff, grp_start, n_groups, cap_groups, cap_entries, hq, err=None, stream=None):
    _check(lib().moe_swiglu_q8_1(_dp(gu), n_ff, _dp(grp_start), _dp(n_groups), cap_groups, cap_entries, _dp(hq),
                                 _dp(err), _stream(stream)))


def grouped_down(typ, codebook, n_embd, n_ff, w_table, n_experts, grp_expert, grp_start, n_groups, cap_groups,
                 grid_groups, hq, cap_entries, ent_dst, out, err=None, stream=None):
    _check(lib().moe_grouped_down(_fmt(typ, codebook), n_embd, n_ff, _dp(w_table), n_experts, _dp(grp_expert),
                                  _dp(grp_start), _dp(n_groups), cap_groups, grid_groups, _dp(hq), cap_entries,
                                  _dp(ent_dst), _dp(out), out.shape[0], out.stride(0), _dp(err),
                                  _stream(stream)))


class ExpertCall:
    """Arguments of one moe_expert_grouped call, kept alive with their tensors."""

    def __init__(self, gu_type, gu_codebook, down_type, down_codebook, n_embd, n_ff, w_gu_table, w_down_table,
                 n_experts, grp_expert, grp_start, n_groups, cap_groups, grid_groups, cap_entries, xq, ent_src,
                 ent_dst, gu, hq, out, err=None, flags=F_PDL):
        self._keep = (gu_codebook, down_codebook, w_gu_table, w_down_table, grp_expert, grp_start, n_groups, xq,
                      ent_src, ent_dst, gu, hq, out, err)
        self.c = ExpertCallC(
            _fmt(gu_type, gu_codebook), _fmt(down_type, down_codebook), n_embd, n_ff, n_experts,
            w_gu_table.data_ptr(), w_down_table.data_ptr(), grp_expert.data_ptr(), grp_start.data_ptr(),
            n_groups.data_ptr(), cap_groups, grid_groups, cap_entries, xq.data_ptr(), xq.shape[0],
            ent_src.data_ptr(), ent_dst.data_ptr(), gu.data_ptr(), hq.data_ptr(), out.data_ptr(), out.shape[0],
            out.stride(0), None if err is None else err.data_ptr(), flags)

    def __call__(self, stream=None):
        _check(lib().moe_expert_grouped(ctypes.byref(self.c), _stream(stream)))

    def call_fused(self, sync, stream=None):
        """The same call in one fused launch (moe_expert_grouped_fused); sync: int32 device tensor
        of grouped_fused_sync_ints(cap_groups, cap_entries, n_ff) words, zeroed before the first
        call (flags MOE_F_SYNC_PAIR / MOE_F_SYNC_ODD in self.c.flags select its halves)."""
        _check(lib().moe_expert_grouped_fused(ctypes.byref(self.c), _dp(sync), _stream(stream)))

    def call_static(self, stream=None):
        """The same call through moe_expert_grouped_static: gu/hq are ignored and the library's
        static device scratch buffer is used instead (nothing is allocated)."""
        _check(lib().moe_expert_grouped_static(ctypes.byref(self.c), _stream(stream)))


def stage_blobs(host_blobs, dev_slots, stream=None):
    """Copy host-resident blobs (uint8 CPU tensors, pinned for the copy kernel) into device staging
    slots (uint8 CUDA tensors, at least as large) with moe_stage_blobs."""
    n = len(host_blobs)
    assert len(dev_slots) == n and all(d.numel() >= h.numel() for h, d in zip(host_blobs, dev_slots))
    src = (ctypes.c_void_p * n)(*[h.data_ptr() for h in host_blobs])
    dst = (ctypes.c_void_p * n)(*[d.data_ptr() for d in dev_slots])
    by = (ctypes.c_int64 * n)(*[h.numel() * h.element_size() for h in host_blobs])
    _check(lib().moe_stage_blobs(src, dst, by, n, _stream(stream)))


def grouped_fused_sync_ints(cap_groups: int, cap_entries: int, n_ff: int) -> int:
    """int32 sync words a moe_expert_grouped_fused call needs (zero them before the first call)."""
    return int(lib().moe_grouped_fused_sync_ints(cap_groups, cap_entries, n_ff))


def layer_sync_ints(T: int, k: int, n_ff: int) -> int:
    """int32 sync words a moe_expert_layer call needs: counters, the call epoch and the flagged h
    copies (zero them once before the first call; torch allocations are 8-byte aligned)."""
    return int(lib().moe_layer_sync_ints(T, k, n_ff))


class LayerCall:
    """Arguments of one moe_expert_layer call (the whole layer in one launch), kept alive with their
    tensors. topk_ids int32 [T, k], x fp32 [T, n_embd], out fp32 [T*k, >= n_embd]; gu / hq scratch
    as for ExpertCall; sync int32 [layer_sync_ints(T, k, n_ff)] zeroed before the first call.
    grp_expert .. xq: optional tensors that receive the grouping and the activation q8_1."""

    def __init__(self, gu_type, gu_codebook, down_type, down_codebook, n_embd, n_ff, w_gu_table, w_down_table,
                 n_experts, topk_ids, x, out, gu, hq, sync, err=None, flags=F_PDL, grp_expert=None, grp_start=None,
                 n_groups=None, ent_src=None, ent_dst=None, xq=None):
        T, k = topk_ids.shape
        opt = (grp_expert, grp_start, n_groups, ent_src, ent_dst, xq)
        self._keep = (gu_codebook, down_codebook, w_gu_table, w_down_table, topk_ids, x, out, gu, hq, sync,
                      err) + opt
        ptr = lambda t: None if t is None else t.data_ptr()
        self.c = LayerCallC(
            _fmt(gu_type, gu_codebook), _fmt(down_type, down_codebook), n_embd, n_ff, n_experts,
            w_gu_table.data_ptr(), w_down_table.data_ptr(), topk_ids.data_ptr(), T, k, x.data_ptr(),
            out.data_ptr(), out.stride(0), gu.data_ptr(), hq.data_ptr(), sync.data_ptr(),
            *[ptr(t) for t in opt], ptr(err), flags)

    def __call__(self, stream=None):
        _check(lib().moe_expert_layer(ctypes.byref(self.c), _stream(stream)))


def router_topk(logits, k, topk_ids=None, weights=None, stream=None):
    """logits fp32 [T, n_experts] -> (topk_ids int32 [T, k], weights fp32 [T, k]) on the device."""
    T, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if weights is None:
        weights = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().moe_router_topk(_dp(logits), T, E, k, _dp(topk_ids), _dp(weights), _stream(stream)))
    return topk_ids, weights


def combine(out, topk_ids, weights, n_experts, y=None, stream=None):
    """out fp32 [T*k, >= n_embd] (row t*k + j = entry (t, j)); -> y fp32 [T, n_embd]."""
    T, k = topk_ids.shape
    N = out.shape[1]
    if y is None:
        y = torch.empty((T, N), dtype=torch.float32, device=out.device)
    _check(lib().moe_combine(_dp(out), out.stride(0), _dp(topk_ids), _dp(weights), T, k, n_experts, N, _dp(y),
                             y.stride(0), _stream(stream)))
    return y


def qsa_block_scores(q, keys, key_scale, scores=None, stream=None):
    """QSA decode block scores: q fp32 [T, 4, 128] (T <= 4), keys int8 [n_blocks, 128], key_scale
    fp32 [n_blocks] -> scores fp32 [T, n_blocks] on the device (the tail block + 1e9)."""
    T = q.shape[0]
    nb = keys.shape[0]
    if scores is None:
        scores = torch.empty((T, nb), dtype=torch.float32, device=q.device)
    _check(lib().moe_qsa_block_scores(_dp(q), T, _dp(keys), _dp(key_scale), nb, _dp(scores), _stream(stream)))
    return scores


def expert_grouped(*args, stream=None, **kw):
    ExpertCall(*args, **kw)(stream)


def transcode_cb(src_type, codebook, dst_type, K, rows, src_table, dst_table, err=None, stream=None):
    """Load-time transcoding of CB2/CB3 blobs (device pointer tables) into slot layouts."""
    _check(lib().moe_transcode_cb(_fmt(src_type, codebook), dst_type, K, rows, src_table.shape[0], _dp(src_table),
                                  _dp(dst_table), _dp(err), _stream(stream)))


def test_block_isum(typ, codebook, K, blob, rows, xq_row, isum, stream=None):
    """Test hook: per-block integer sums of `rows` rows of `blob` against one q8_1 row."""
    _check(lib().moe_test_block_isum(_fmt(typ, codebook), K, _dp(blob), rows, _dp(xq_row), _dp(isum),
                                     _stream(stream)))
