"""Python face of the CPU oracle (oracle.c) for the grouped routed-expert decode.

TEST INFRASTRUCTURE, NOT THE PRODUCT: only tests/, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import this package. It compiles oracle.c
with gcc (``-O2 -ffp-contract=off``, no fast-math) into ``oracle/_build/`` and calls it with
ctypes; it shares no code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict = {}

Q8_0, Q4B, NL4, CB2, CB3, CB3X, CB2X = 1, 2, 3, 4, 5, 6, 7
TYPE_NAMES = {"Q8_0": Q8_0, "Q4B": Q4B, "NL4": NL4, "CB2": CB2, "CB3": CB3, "CB3X": CB3X, "CB2X": CB2X}

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64


def build(defines=()) -> str:
    """Compile oracle.c (with optional planted-mistake macros) and return the .so path."""
    tag = "_".join(sorted(defines)) or "base"
    out = os.path.join(_BUILD, f"liboracle_{tag}.so")
    src = os.path.join(_HERE, "oracle.c")
    if os.path.exists(out) and os.path.getmtime(out) >= max(
        os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, src, "-lm"] + [f"-D{d}" for d in defines]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _setup(lib):
    lib.orc_h2f.argtypes = [ctypes.c_uint16]
    lib.orc_h2f.restype = ctypes.c_float
    lib.orc_f2h.argtypes = [ctypes.c_float]
    lib.orc_f2h.restype = ctypes.c_uint16
    for f in ("orc_expf", "orc_silu"):
        getattr(lib, f).argtypes = [ctypes.c_float]
        getattr(lib, f).restype = ctypes.c_float
    lib.orc_swiglu.argtypes = [ctypes.c_float, ctypes.c_float]
    lib.orc_swiglu.restype = ctypes.c_float
    lib.orc_row_bytes.argtypes = [_I, _I]
    lib.orc_row_bytes.restype = _I64
    lib.orc_quantize_q8_1.argtypes = [_P, _I64, _P]
    lib.orc_dequant_row.argtypes = [_I, _P, _I, _P, _P]
    lib.orc_int_weights.argtypes = [_I, _P, _I, _P, _P]
    lib.orc_block_isum.argtypes = [_I, _P, _I, _P, _P, _P]
    lib.orc_row_dot.argtypes = [_I, _P, _I, _P, _P]
    lib.orc_row_dot.restype = ctypes.c_double
    lib.orc_grouped_gemv.argtypes = [_I, _P, _I, _I, _P, _I, _P, _P, _I, _P, _P, _P, _P, _I64]
    lib.orc_grouped_gemv.restype = _I
    lib.orc_swiglu_q8_1.argtypes = [_P, _I, _I, _I, _P]
    lib.orc_transcode_row.argtypes = [_I, _P, _I, _P, _I, _P]
    lib.orc_transcode_row.restype = _I
    lib.orc_route_group.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P]
    lib.orc_router_topk.argtypes = [_P, _I, _I, _I, _P, _P]
    lib.orc_router_topk.restype = _I
    lib.orc_combine.argtypes = [_P, _I64, _P, _P, _I, _I, _I, _I, _P]
    lib.orc_route_group.restype = _I
    lib.orc_qsa_block_scores.argtypes = [_P, _I, _P, _P, _I64, _P]
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """numpy wrappers over one build of oracle.c."""

    def __init__(self, defines=()):
        with _LOCK:
            key = tuple(sorted(defines))
            if key not in _LIBS:
                _LIBS[key] = _setup(ctypes.CDLL(build(defines)))
            self.lib = _LIBS[key]

    # ---- scalars
    def h2f(self, h):
        h = np.asarray(h, dtype=np.uint16).ravel()
        return np.array([self.lib.orc_h2f(int(v)) for v in h], dtype=np.float32)

    def f2h(self, f):
        f = np.asarray(f, dtype=np.float32).ravel()
        return np.array([self.lib.orc_f2h(float(v)) for v in f], dtype=np.uint16)

    def expf(self, x):
        x = np.asarray(x, dtype=np.float32).ravel()
        return np.array([self.lib.orc_expf(float(v)) for v in x], dtype=np.float32)

    def silu(self, x):
        x = np.asarray(x, dtype=np.float32).ravel()
        return np.array([self.lib.orc_silu(float(v)) for v in x], dtype=np.float32)

    def swiglu(self, g, u):
        g = np.asarray(g, dtype=np.float32).ravel()
        u = np.asarray(u, dtype=np.float32).ravel()
        return np.array([self.lib.orc_swiglu(float(a), float(b)) for a, b in zip(g, u)], dtype=np.float32)

    # ---- q8_1
    def row_bytes(self, typ, K):
        return int(self.lib.orc_row_bytes(typ, K))

    def quantize_q8_1(self, x):
        """x: float32 [rows, cols] -> uint8 [rows, cols/32, 36]."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        rows, cols = x.shape
        out = np.zeros((rows, cols // 32, 36), dtype=np.uint8)
        self.lib.orc_quantize_q8_1(_ptr(x), x.size, _ptr(out))
        return out

    # ---- rows
    def _cb(self, cb):
        return None if cb is None else np.ascontiguousarray(cb, dtype=np.int8)

    def dequant_row(self, typ, row, K, cb=None):
        row = np.ascontiguousarray(row, dtype=np.uint8)
        cb = self._cb(cb)
        w = np.zeros(K, dtype=np.float64)
        self.lib.orc_dequant_row(typ, _ptr(row), K, _ptr(cb), _ptr(w))
        return w

    def int_weights(self, typ, row, K, cb=None):
        row = np.ascontiguousarray(row, dtype=np.uint8)
        cb = self._cb(cb)
        v = np.zeros(K, dtype=np.int32)
        self.lib.orc_int_weights(typ, _ptr(row), K, _ptr(cb), _ptr(v))
        return v

    def block_isum(self, typ, row, K, xq_row, cb=None):
        row = np.ascontiguousarray(row, dtype=np.uint8)
        xq_row = np.ascontiguousarray(xq_row, dtype=np.uint8)
        cb = self._cb(cb)
        out = np.zeros(K // 32, dtype=np.int32)
        self.lib.orc_block_isum(typ, _ptr(row), K, _ptr(cb), _ptr(xq_row), _ptr(out))
        return out

    def row_dot(self, typ, row, K, xq_row, cb=None):
        row = np.ascontiguousarray(row, dtype=np.uint8)
        xq_row = np.ascontiguousarray(xq_row, dtype=np.uint8)
        cb = self._cb(cb)
        return float(self.lib.orc_row_dot(typ, _ptr(row), K, _ptr(cb), _ptr(xq_row)))

    def transcode_row(self, src_type, row, K, cb, dst_type):
        row = np.ascontiguousarray(row, dtype=np.uint8)
        cb = self._cb(cb)
        out = np.zeros(self.row_bytes(dst_type, K), dtype=np.uint8)
        rc = self.lib.orc_transcode_row(src_type, _ptr(row), K, _ptr(cb), dst_type, _ptr(out))
        return out, rc

    def transcode_blob(self, src_type, blob, K, rows, cb, dst_type):
        rb_s, rb_d = self.row_bytes(src_type, K), self.row_bytes(dst_type, K)
        out = np.zeros(rows * rb_d, dtype=np.uint8)
        bad = 0
        for r in range(rows):
            o, rc = self.transcode_row(src_type, blob[r * rb_s:(r + 1) * rb_s], K, cb, dst_type)
            out[r * rb_d:(r + 1) * rb_d] = o
            bad |= rc
        return out, bad

    # ---- grouped steps
    def grouped_gemv(self, typ, K, rows, blobs, grp_expert, grp_start, n_groups, act,
                     ent_in=None, ent_out=None, out=None, cb=None):
        """blobs: list of uint8 arrays (one per expert); act: uint8 [n_rows, K/32, 36];
        out: float64 [n_out_rows, rows] (updated in place and returned)."""
        cb = self._cb(cb)
        blobs = [np.ascontiguousarray(b, dtype=np.uint8) for b in blobs]
        ptrs = (ctypes.c_void_p * len(blobs))(*[b.ctypes.data for b in blobs])
        ge = np.ascontiguousarray(grp_expert, dtype=np.int32)
        gs = np.ascontiguousarray(grp_start, dtype=np.int32)
        act = np.ascontiguousarray(act, dtype=np.uint8)
        ei = None if ent_in is None else np.ascontiguousarray(ent_in, dtype=np.int32)
        eo = None if ent_out is None else np.ascontiguousarray(ent_out, dtype=np.int32)
        assert out is not None and out.dtype == np.float64 and out.flags.c_contiguous
        rc = self.lib.orc_grouped_gemv(typ, _ptr(cb), K, rows, ptrs, len(blobs), _ptr(ge), _ptr(gs),
                                       int(n_groups), _ptr(act), _ptr(ei), _ptr(eo), _ptr(out),
                                       out.shape[1])
        return out, rc

    def swiglu_q8_1(self, gu, F, e0, e1, hq):
        gu = np.ascontiguousarray(gu, dtype=np.float32)
        assert hq.dtype == np.uint8 and hq.flags.c_contiguous
        self.lib.orc_swiglu_q8_1(_ptr(gu), F, int(e0), int(e1), _ptr(hq))
        return hq

    def router_topk(self, logits, k):
        """logits fp32 [T, E] -> (topk_ids int32 [T, k], weights fp64 [T, k], rc)."""
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        ids = np.zeros((T, k), np.int32)
        w = np.zeros((T, k), np.float64)
        rc = self.lib.orc_router_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w))
        return ids, w, rc

    def combine(self, out, topk_ids, weights, n_experts):
        """out fp32 [T*k, n_embd]; topk_ids [T, k]; weights [T, k] -> y fp64 [T, n_embd]."""
        out = np.ascontiguousarray(out, dtype=np.float32)
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        w = np.ascontiguousarray(weights, dtype=np.float64)
        T, k = ids.shape
        y = np.zeros((T, out.shape[1]), np.float64)
        self.lib.orc_combine(_ptr(out), out.shape[1], _ptr(ids), _ptr(w), T, k, int(n_experts), out.shape[1], _ptr(y))
        return y

    def qsa_block_scores(self, q, keys, scale):
        """q fp32 [T, 4, 128]; keys int8 [n_blocks, 128]; scale fp32 [n_blocks] -> scores fp32
        [T, n_blocks] (QSA decode block scores, the tail block + 1e9)."""
        q = np.ascontiguousarray(q, dtype=np.float32)
        keys = np.ascontiguousarray(keys, dtype=np.int8)
        scale = np.ascontiguousarray(scale, dtype=np.float32)
        T = q.shape[0]
        assert q.shape[1:] == (4, 128) and keys.shape[1] == 128 and scale.shape == (keys.shape[0],)
        out = np.zeros((T, keys.shape[0]), np.float32)
        self.lib.orc_qsa_block_scores(_ptr(q), T, _ptr(keys), _ptr(scale), keys.shape[0], _ptr(out))
        return out

    def route_group(self, topk_ids, n_experts, entry_base=0, cap_entries=None):
        ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        T, k = ids.shape
        n = T * k
        cap_entries = cap_entries or entry_base + n
        ge = np.full(n + 1, -1, dtype=np.int32)
        gs = np.full(n + 2, -1, dtype=np.int32)
        ng = np.zeros(1, dtype=np.int32)
        es = np.full(cap_entries, -1, dtype=np.int32)
        ed = np.full(cap_entries, -1, dtype=np.int32)
        dropped = self.lib.orc_route_group(_ptr(ids), T, k, n_experts, entry_base, _ptr(ge), _ptr(gs),
                                           _ptr(ng), _ptr(es), _ptr(ed))
        G = int(ng[0])
        return dict(grp_expert=ge[:G], grp_start=gs[:G + 1], n_groups=G, ent_src=es, ent_dst=ed,
                    dropped=int(dropped))


_DEFAULT = None


def get() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
