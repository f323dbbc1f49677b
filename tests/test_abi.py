"""The C-ABI library on the CPU: it loads, exports every entry point the headers declare, and
rejects bad host-visible arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    from quantized_routed_expert_grouped_gb300 import build
    build.build()
    import quantized_routed_expert_grouped_gb300 as mod
    mod.lib()
    return mod


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*(?:int|int64_t|const char\*)\s+(moe_\w+)\s*\(", src, re.M))
    return sorted(names)


def test_exports_every_declared_symbol(m):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(m.lib(), n), n


def test_row_bytes_and_strerror(m):
    assert m.row_bytes(m.CB3, 2560) == 1020 and m.row_bytes(m.CB2, 2560) == 700
    assert m.row_bytes(m.NL4, 768) == 432 and m.row_bytes(m.Q8_0, 512) == 544 and m.row_bytes(m.Q4B, 4096) == 2560
    assert m.row_bytes(m.CB3, 100) == 0 and m.row_bytes(99, 256) == 0
    assert "shape" in m.strerror(-3)


def test_host_argument_errors(m):
    L = m.lib()
    W = m.WFmt
    dummy = ctypes.c_void_p(16)
    # unsupported type, missing codebook, bad shape, NULL pointers, bad capacities
    assert L.moe_grouped_gu(W(9, None), 2560, 768, dummy, 1, dummy, dummy, dummy, 1, 0, dummy, 1, dummy, 1, dummy,
                            None, None) == -2
    assert L.moe_grouped_gu(W(5, None), 2560, 768, dummy, 1, dummy, dummy, dummy, 1, 0, dummy, 1, dummy, 1, dummy,
                            None, None) == -2
    assert L.moe_grouped_gu(W(1, None), 2500, 768, dummy, 1, dummy, dummy, dummy, 1, 0, dummy, 1, dummy, 1, dummy,
                            None, None) == -3
    assert L.moe_grouped_gu(W(1, None), 2560, 768, None, 1, dummy, dummy, dummy, 1, 0, dummy, 1, dummy, 1, dummy,
                            None, None) == -1
    assert L.moe_grouped_gu(W(1, None), 2560, 768, dummy, 0, dummy, dummy, dummy, 1, 0, dummy, 1, dummy, 1, dummy,
                            None, None) == -4
    assert L.moe_grouped_down(W(3, None), 2560, 768, dummy, 1, dummy, dummy, dummy, 1, 0, dummy, 1, dummy, dummy,
                              4, 2560, None, None) == -2
    assert L.moe_grouped_down(W(1, None), 2560, 768, dummy, 1, dummy, dummy, dummy, 1, 0, dummy, 1, dummy, dummy,
                              4, 100, None, None) == -3
    assert L.moe_swiglu_q8_1(dummy, 100, dummy, dummy, 1, 1, dummy, None, None) == -3
    assert L.moe_quantize_q8_1(None, 1, 32, dummy, None) == -1
    assert L.moe_quantize_q8_1(dummy, 1, 33, dummy, None) == -3
    assert L.moe_route_group(dummy, 40, 32, 8, 0, dummy, dummy, dummy, dummy, dummy, None, None) == -3
    assert L.moe_expert_grouped(None, None) == -1
    assert L.moe_test_block_isum(W(1, None), 300, dummy, 1, dummy, dummy, None) == -3
    # the router and the combine
    assert L.moe_router_topk(None, 4, 128, 8, dummy, dummy, None) == -1
    assert L.moe_router_topk(dummy, 4, 128, 33, dummy, dummy, None) == -3   # k > 32
    assert L.moe_router_topk(dummy, 4, 4, 8, dummy, dummy, None) == -3      # k > n_experts
    assert L.moe_router_topk(dummy, 4, 2000, 8, dummy, dummy, None) == -3   # n_experts > 1024
    assert L.moe_combine(dummy, 2560, dummy, dummy, 4, 8, 128, 2560, None, 2560, None) == -1
    assert L.moe_combine(dummy, 100, dummy, dummy, 4, 8, 128, 2560, dummy, 2560, None) == -3
    assert L.moe_combine(dummy, 2560, dummy, dummy, 70000, 8, 128, 2560, dummy, 2560, None) == -3
    assert L.moe_combine(dummy, 2560, dummy, dummy, 4, 8, 0, 2560, dummy, 2560, None) == -4
    # QSA block scores
    assert L.moe_qsa_block_scores(None, 4, dummy, dummy, 100, dummy, None) == -1
    assert L.moe_qsa_block_scores(dummy, 5, dummy, dummy, 100, dummy, None) == -3   # T > 4
    assert L.moe_qsa_block_scores(dummy, 0, dummy, dummy, 100, dummy, None) == -3
    assert L.moe_qsa_block_scores(dummy, 4, dummy, dummy, 0, dummy, None) == -3     # no block
    assert L.moe_qsa_block_scores(ctypes.c_void_p(20), 4, dummy, dummy, 100, dummy, None) == -6  # q unaligned


def test_layer_call_host_errors(m):
    L = m.lib()
    W = m.WFmt
    d = 16
    # control words + per entry (32) and h block (24) nine 8-byte pairs
    assert m.layer_sync_ints(4, 8, 768) == 4 + 32 * 24 * 9 * 2
    assert m.layer_sync_ints(0, 8, 768) == 0

    def call(**kw):
        f = dict(gu_fmt=W(1, None), down_fmt=W(1, None), n_embd=2560, n_ff=768, n_experts=4, w_gu=d, w_down=d,
                 topk_ids=d, T=4, k=8, x=d, out=d, out_row_stride=2560, gu=d, hq=d, sync=d, flags=0)
        f.update(kw)
        c = m.LayerCallC(**f)
        return L.moe_expert_layer(ctypes.byref(c), None)

    assert L.moe_expert_layer(None, None) == -1
    assert call(down_fmt=W(4, ctypes.c_void_p(d))) == -2        # CB2 down: not supported by the fused call
    assert call(gu_fmt=W(5, None)) == -2                         # CB3 without codebook
    assert call(n_ff=700) == -3
    assert call(sync=None) == -1 and call(x=None) == -1 and call(topk_ids=None) == -1
    assert call(T=0) == -3
    assert call(T=65) == -4                                      # T*k > 512
    assert call(T=40, k=2) == -4                                 # 40 activation rows exceed the staging budget
    assert call(out_row_stride=100) == -3
    assert call(n_experts=0) == -4 and call(n_experts=(1 << 26) + 1) == -4
    assert call(sync=d + 4) == -6                                 # sync holds 8-byte pairs



def test_fused_grouped_call_and_staging_host_errors(m):
    """The one-launch expert call and the staging copies reject bad host-visible arguments before
    any CUDA call (so these run without a GPU)."""
    L = m.lib()
    W = m.WFmt
    d = 16

    def call(sync=d, **kw):
        f = dict(gu_fmt=W(1, None), down_fmt=W(3, ctypes.c_void_p(d)), n_embd=2560, n_ff=768, n_experts=64,
                 w_gu=d, w_down=d, grp_expert=d, grp_start=d, n_groups=d, cap_groups=32, grid_groups=0,
                 cap_entries=34, xq=d, n_xq_rows=4, ent_src=d, ent_dst=d, gu=d, hq=d, out=d, out_rows=38,
                 out_row_stride=2560, err=None, flags=0)
        f.update(kw)
        c = m.ExpertCallC(**f)
        return L.moe_expert_grouped_fused(ctypes.byref(c), None if sync is None else ctypes.c_void_p(sync), None)

    assert L.moe_expert_grouped_fused(None, ctypes.c_void_p(d), None) == -1
    assert call(sync=None) == -1 and call(grp_start=None) == -1 and call(ent_dst=None) == -1
    assert call(down_fmt=W(4, ctypes.c_void_p(d))) == -2        # CB2 down: not a down format of the fused call
    assert call(n_ff=700) == -3
    assert call(cap_groups=0) == -4 and call(n_xq_rows=0) == -4 and call(out_rows=0) == -4
    assert call(out_row_stride=100) == -3
    assert call(xq=d + 2) == -6 and call(gu=d + 8) == -6 and call(sync=d + 4) == -6
    # staging: n < 0, a NULL blob or slot, a size <= 0, a slot not 16-byte aligned; n = 0 is a no-op
    src = (ctypes.c_void_p * 2)(d, d)
    dst = (ctypes.c_void_p * 2)(32, 48)
    by = (ctypes.c_int64 * 2)(64, 64)
    assert L.moe_stage_blobs(None, None, None, 0, None) == 0
    assert L.moe_stage_blobs(src, dst, by, -1, None) == -3
    assert L.moe_stage_blobs(None, dst, by, 2, None) == -1
    assert L.moe_stage_blobs(src, dst, (ctypes.c_int64 * 2)(64, 0), 2, None) == -3
    assert L.moe_stage_blobs(src, (ctypes.c_void_p * 2)(32, 40), by, 2, None) == -6
    assert L.moe_stage_blobs((ctypes.c_void_p * 2)(d, None), dst, by, 2, None) == -1
