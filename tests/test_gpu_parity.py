"""Parity of the CUDA path (through the C ABI) with the CPU oracle, stage by stage and end to end.

Bars: integer and byte results (q8_1 codes and scales, per-block integer sums, routing and scatter
indices) bit-exact; fp32 outputs within max|err| / max|ref| <= 1e-5 per output row. Inputs come
from the seeded generators; the oracle never takes an input produced by the CUDA path.
"""
import numpy as np
import pytest
import torch

import harness as H
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module")
def m():
    import quantized_routed_expert_grouped_gb300 as mod
    mod.lib()
    return mod


# ------------------------------------------------------------------ a1: activation q8_1

def test_quantize_q8_1_bitexact(m, orc):
    rng = np.random.Generator(np.random.PCG64(1))
    x = rng.standard_normal((7, 4096)).astype(np.float32) * np.exp(rng.uniform(-8, 8, (7, 1))).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 20
    x[0, :32] = 0.0                      # zero block
    x[1, :32] = 3.0                      # constant block
    x[2, :8] = [127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5]  # halfway cases
    x[2, 8:32] = 0
    got = m.quantize_q8_1(torch.from_numpy(x).cuda()).cpu().numpy()
    assert np.array_equal(got, orc.quantize_q8_1(x))


# ------------------------------------------------------------------ a2/a4 integer block sums

@pytest.mark.parametrize("typ", [synth.Q8_0, synth.Q4B, synth.NL4, synth.CB2, synth.CB3, synth.CB3X, synth.CB2X])
@pytest.mark.parametrize("K", [256, 768, 2560, 8192])
def test_block_isum_bitexact(m, orc, typ, K):
    rows = 24
    src = {synth.CB3X: synth.CB3, synth.CB2X: synth.CB2}.get(typ, typ)
    blob = synth.weight_blobs(src, rows, K, 1, synth.derive_key(src, K), "cpu")[0]
    cb = synth.codebook(src, K + src)
    if src != typ:  # slot layouts: the oracle's own transcoding of the native blob
        t, rc = orc.transcode_blob(src, blob.numpy(), K, rows, cb, typ)
        assert rc == 0
        blob, cb = torch.from_numpy(t), None
    x = synth.activations(1, K, K * 3 + typ, outliers=0.01)
    xq = orc.quantize_q8_1(x)
    pad = torch.zeros(blob.numel() + 64, dtype=torch.uint8)
    pad[:blob.numel()] = blob
    cbd = None if cb is None else torch.from_numpy(np.ascontiguousarray(cb).ravel()).cuda()
    isum = torch.zeros((rows, K // 32), dtype=torch.int32, device="cuda")
    m.test_block_isum(typ, cbd, K, pad.cuda(), rows, torch.from_numpy(xq).cuda(), isum)
    got = isum.cpu().numpy()
    rb = synth.row_bytes(typ, K)
    b = blob.numpy()
    for r in range(rows):
        want = orc.block_isum(typ, b[r * rb:(r + 1) * rb], K, xq[0], cb)
        assert np.array_equal(got[r], want), (r, np.nonzero(got[r] != want))


# ------------------------------------------------------------------ load-time transcoding

# rows: one run of whole rows per CTA (256 / (K / 256) rows), so 60 rows of K = 2560 take three
# CTAs (25, 25, 10) and 100 rows of K = 768 two (85, 15)
@pytest.mark.parametrize("src,dst,K,rows", [(synth.CB3, synth.CB3X, 2560, 16), (synth.CB2, synth.CB2X, 768, 16),
                                            (synth.CB2, synth.CB3X, 512, 16), (synth.CB3, synth.CB3X, 768, 16),
                                            (synth.CB3, synth.CB3X, 2560, 60), (synth.CB2, synth.CB2X, 768, 100)])
def test_transcode_bitexact(m, orc, src, dst, K, rows):
    nb = 3
    blobs = synth.weight_blobs(src, rows, K, nb, synth.derive_key(src, dst, K), "cuda")
    cb = synth.codebook(src, 5 + K)
    cbd = torch.from_numpy(np.ascontiguousarray(cb).ravel()).cuda()
    out = torch.zeros((nb, rows * synth.row_bytes(dst, K)),
                      dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.transcode_cb(src, cbd, dst, K, rows, H.pointer_table(blobs), H.pointer_table(out), err)
    got = out.cpu().numpy()
    assert int(err.item()) == 0
    for b in range(nb):
        want, rc = orc.transcode_blob(src, blobs[b].cpu().numpy(), K, rows, cb, dst)
        assert rc == 0 and np.array_equal(got[b], want), b
    # a grid value outside the slot's range is reported
    bad = cb.copy()
    bad.ravel()[0] = 17 if dst == synth.CB3X else 5
    m.transcode_cb(src, torch.from_numpy(np.ascontiguousarray(bad).ravel()).cuda(), dst, K, rows,
                   H.pointer_table(blobs), H.pointer_table(out), err)
    assert int(err.item()) & 32
    # a destination pointer off the 8-byte boundary: that blob is reported and left unwritten (the
    # offset keeps every byte the kernel could write inside the buffer)
    out.zero_()
    err.zero_()
    tab = H.pointer_table(out)
    tab[0] += 4
    m.transcode_cb(src, cbd, dst, K, rows, H.pointer_table(blobs), tab, err)
    got = out.cpu().numpy()
    assert int(err.item()) == 16
    assert not got[0].any()
    for b in range(1, nb):
        want, _ = orc.transcode_blob(src, blobs[b].cpu().numpy(), K, rows, cb, dst)
        assert np.array_equal(got[b], want), b


# ------------------------------------------------------------------ a0: routing

@pytest.mark.parametrize("T,k,E,base", [(1, 2, 8, 0), (4, 8, 64, 0), (4, 8, 128, 3), (3, 8, 16, 0), (32, 32, 40, 7)])
def test_route_group_bitexact(m, orc, T, k, E, base):
    ids = synth.routing(T, k, E, T * 100 + k + E)
    r = orc.route_group(ids, E, entry_base=base)
    n = T * k
    ge = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    gs = torch.full((n + 1,), -7, dtype=torch.int32, device="cuda")
    ng = torch.zeros(1, dtype=torch.int32, device="cuda")
    es = torch.full((base + n,), -7, dtype=torch.int32, device="cuda")
    ed = torch.full((base + n,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.route_group(torch.from_numpy(ids).cuda(), E, base, ge, gs, ng, es, ed, err)
    G = r["n_groups"]
    assert int(ng.item()) == G and int(err.item()) == 0
    assert np.array_equal(ge.cpu().numpy()[:G], r["grp_expert"])
    assert np.array_equal(gs.cpu().numpy()[:G + 1], r["grp_start"])
    assert np.array_equal(es.cpu().numpy()[base:], r["ent_src"][base:])
    assert np.array_equal(ed.cpu().numpy()[base:], r["ent_dst"][base:])
    assert (es.cpu().numpy()[:base] == -7).all()


def test_route_group_drops_bad_ids(m, orc):
    ids = np.array([[3, 9, -1], [2, 3, 1]], np.int32)
    r = orc.route_group(ids, 8)
    ge = torch.full((6,), -7, dtype=torch.int32, device="cuda")
    gs = torch.full((7,), -7, dtype=torch.int32, device="cuda")
    ng = torch.zeros(1, dtype=torch.int32, device="cuda")
    es = torch.full((6,), -7, dtype=torch.int32, device="cuda")
    ed = torch.full((6,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.route_group(torch.from_numpy(ids).cuda(), 8, 0, ge, gs, ng, es, ed, err)
    G = r["n_groups"]
    assert int(ng.item()) == G and int(err.item()) & 128
    assert np.array_equal(gs.cpu().numpy()[:G + 1], r["grp_start"])
    assert np.array_equal(es.cpu().numpy()[:4], r["ent_src"][:4])


# ------------------------------------------------------------------ a3: SwiGLU + q8_1 on synthetic gate/up

@pytest.mark.parametrize("F", [256, 768, 1536])
def test_swiglu_q8_1_bitexact(m, orc, F):
    rng = np.random.Generator(np.random.PCG64(F))
    cap = 40
    gu = (rng.standard_normal((cap, 2 * F)) * np.exp(rng.uniform(-3, 3, (cap, 1)))).astype(np.float32)
    gu[5, :] = 0.0
    gu[6, :F] = -200.0
    gs = np.array([9, 12, 20, 29], np.int32)   # entries [9, 29) over 3 groups
    hq = torch.full((cap, F // 32, 36), 0xA5, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ng = torch.tensor([3], dtype=torch.int32, device="cuda")
    m.swiglu_q8_1(torch.from_numpy(gu).cuda(), F, torch.from_numpy(gs).cuda(), ng, 8, cap, hq, err)
    want = np.full((cap, F // 32, 36), 0xA5, np.uint8)
    orc.swiglu_q8_1(gu, F, 9, 29, want)
    assert np.array_equal(hq.cpu().numpy(), want)
    assert int(err.item()) == 0


# ------------------------------------------------------------------ a2 + a3 + a4 stage by stage

def _stage_inputs(orc, L, r):
    """Oracle-made q8_1 activations and an oracle-made hq from synthetic h (not from the GPU)."""
    wl = L.wl
    xq = orc.quantize_q8_1(L.x)
    n = L.T * wl.k
    rng = np.random.Generator(np.random.PCG64(L.layer + 99))
    h = rng.standard_normal((n, wl.F)).astype(np.float32)
    hq = orc.quantize_q8_1(h)
    return xq, hq


# (workload, (gate/up, down), T, slot layout the gate/up pool is transcoded to or None)
CASES = [("tiny", (synth.Q8_0, synth.Q8_0), 1, None), ("verify", (synth.CB2, synth.NL4), 4, None),
         ("window48", (synth.CB3, synth.NL4), 1, None), ("window48", (synth.CB3, synth.NL4), 3, None),
         ("window48", (synth.CB3, synth.NL4), 4, synth.CB3X), ("verify", (synth.CB2, synth.NL4), 4, synth.CB2X),
         # T > 4: groups of up to T entries, several 4-entry batches per weight tile
         ("verify", (synth.CB2, synth.NL4), 8, None), ("window48", (synth.CB3, synth.NL4), 6, synth.CB3X)]
CASE_IDS = [f"{c[0]}-T{c[2]}" + (f"-{synth.NAMES[c[3]]}" if c[3] else "") for c in CASES]


@pytest.mark.parametrize("wname,pair,T,xt", CASES, ids=CASE_IDS)
def test_grouped_stages(m, orc, wname, pair, T, xt):
    wl = synth.WORKLOADS[wname]
    L0 = H.make_layer(wl, pair, T)
    L = H.transcoded(m, L0, xt) if xt else L0
    r = orc.route_group(L.ids, wl.E)
    G, n = r["n_groups"], T * wl.k
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    xq, hq = _stage_inputs(orc, L, r)
    # gate/up on oracle-made xq
    xq_d = torch.from_numpy(xq).cuda()
    m.grouped_gu(L.gu_t, L.cb_gu_d, wl.N, wl.F, L.tab_gu, wl.E, B.grp_expert, B.grp_start, B.n_groups,
                 B.cap_groups, 0, xq_d, B.ent_src, B.cap_entries, B.gu, B.err)
    gub = H.host_blobs(L0, r["grp_expert"], "gu")
    ref = np.full((n, 2 * wl.F), np.nan)
    orc.grouped_gemv(L0.gu_t, wl.N, 2 * wl.F, gub, r["grp_expert"], r["grp_start"], G, xq, ent_in=r["ent_src"],
                     out=ref, cb=L0.cb_gu)
    got = B.gu.cpu().numpy()
    assert H.rel_err(got, ref) <= TOL
    # down on oracle-made hq, scattered destinations
    hq_d = torch.from_numpy(hq).cuda()
    m.grouped_down(L.dn_t, L.cb_dn_d, wl.N, wl.F, L.tab_dn, wl.E, B.grp_expert, B.grp_start, B.n_groups,
                   B.cap_groups, 0, hq_d, B.cap_entries, B.ent_dst, B.out, B.err)
    dnb = H.host_blobs(L, r["grp_expert"], "dn")
    ref = np.full((n, wl.N), np.nan)
    orc.grouped_gemv(L.dn_t, wl.F, wl.N, dnb, r["grp_expert"], r["grp_start"], G, hq, ent_out=r["ent_dst"],
                     out=ref, cb=L.cb_dn)
    got = B.out.cpu().numpy()
    assert H.rel_err(got, ref) <= TOL
    assert int(B.err.item()) == 0


# ------------------------------------------------------------------ end to end, grid invariance, untouched rows

def _e2e(m, orc, L, grid_groups=0, flags=1):
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    H.expert_call(m, L, B, grid_groups, flags)()
    torch.cuda.synchronize()
    return B


@pytest.mark.parametrize("wname,pair,T,xt", CASES, ids=CASE_IDS)
def test_expert_grouped_end_to_end(m, orc, wname, pair, T, xt):
    wl = synth.WORKLOADS[wname]
    L0 = H.make_layer(wl, pair, T)
    L = H.transcoded(m, L0, xt) if xt else L0
    ref = H.oracle_call(orc, L0)
    B = _e2e(m, orc, L)
    assert int(B.err.item()) == 0
    assert np.array_equal(B.xq.cpu().numpy(), ref["xq"])
    assert H.rel_err(B.gu.cpu().numpy(), ref["gu"]) <= TOL
    flips, scale_diffs = H.q8_1_code_flips(B.hq.cpu().numpy(), ref["hq"])
    n = T * wl.k
    assert flips <= max(2, n * wl.F // 4096) and scale_diffs <= 2, (flips, scale_diffs)
    err = H.rel_err(B.out.cpu().numpy(), ref["out"])
    assert err <= (TOL if flips == 0 and scale_diffs == 0 else 2e-3), (err, flips)


def test_grid_invariance_and_pdl(m, orc):
    wl = synth.WORKLOADS["verify"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    base = _e2e(m, orc, L, 0)
    for gg in (1, 2, 3, 4, 33, 1000):
        for flags in (0, 1):
            B = _e2e(m, orc, L, gg, flags)
            assert torch.equal(B.gu.view(torch.int32), base.gu.view(torch.int32)), gg
            assert torch.equal(B.hq, base.hq), gg
            assert torch.equal(B.out.view(torch.int32), base.out.view(torch.int32)), gg


def test_empty_call_writes_nothing(m, orc):
    wl = synth.WORKLOADS["verify"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    B.n_groups.zero_()
    for gg in (0, 1, 4):
        H.expert_call(m, L, B, gg)()
    torch.cuda.synchronize()
    assert torch.isnan(B.gu).all() and torch.isnan(B.out).all() and (B.hq == 0xA5).all()
    assert int(B.err.item()) == 0


def test_second_call_after_first(m, orc):
    """A second call per layer (the PCIe call of #363): n_groups in {0, 1}, 1-2 entries numbered
    after the first call's, scattered destinations; rows it does not own stay NaN."""
    wl = synth.WORKLOADS["sparse"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    n = L.T * wl.k
    xq = orc.quantize_q8_1(L.x)
    gub = H.host_blobs(L, [5, 17], "gu")
    dnb = H.host_blobs(L, [5, 17], "dn")
    for ng, ne in ((0, 0), (1, 1), (1, 2)):
        cap_e = n + 2
        B = H.make_bufs(L, cap_entries=cap_e, out_rows=n + 6)
        m.quantize_q8_1(torch.from_numpy(L.x).cuda(), B.xq)
        ge = np.array([17] + [0] * (n - 1), np.int32)
        gs = np.array([n, n + ne] + [0] * (n - 1), np.int32)
        es = np.full(cap_e, -7, np.int32); es[n:n + ne] = [3, 1][:ne]
        ed = np.full(cap_e, -7, np.int32); ed[n:n + ne] = [n + 4, 2][:ne]
        B.grp_expert.copy_(torch.from_numpy(ge)); B.grp_start.copy_(torch.from_numpy(gs))
        B.n_groups.fill_(ng)
        B.ent_src.copy_(torch.from_numpy(es)); B.ent_dst.copy_(torch.from_numpy(ed))
        for gg in (0, 1, 2, 3, 4, 33):
            B.gu.fill_(float("nan")); B.out.fill_(float("nan")); B.hq.fill_(0xA5)
            H.expert_call(m, L, B, gg)()
            torch.cuda.synchronize()
            gu = B.gu.cpu().numpy(); out = B.out.cpu().numpy(); hq = B.hq.cpu().numpy()
            assert int(B.err.item()) == 0
            own_gu = set(range(n, n + ne)) if ng else set()
            own_out = set(ed[n:n + ne].tolist()) if ng else set()
            for i in range(cap_e):
                assert np.isnan(gu[i]).all() == (i not in own_gu)
                assert (hq[i] == 0xA5).all() == (i not in own_gu)
            for i in range(n + 6):
                assert np.isnan(out[i]).all() == (i not in own_out)
            if ng:
                # the oracle's chain for this call's one group: gate/up (fp64) ...
                ref = np.full((cap_e, 2 * wl.F), np.nan)
                orc.grouped_gemv(L.gu_t, wl.N, 2 * wl.F, gub, ge[:1], gs[:2], 1, xq, ent_in=es, out=ref, cb=L.cb_gu)
                assert H.rel_err(gu[n:n + ne], ref[n:n + ne]) <= TOL
                # ... SwiGLU + q8_1 over the call's own entries: bit for bit on the GPU's gate/up
                # rows (same fp32 inputs), then on the oracle's own fp32-rounded rows ...
                hq_stage = np.zeros((cap_e, wl.F // 32, 36), np.uint8)
                orc.swiglu_q8_1(gu, wl.F, n, n + ne, hq_stage)
                assert (hq[n:n + ne] == hq_stage[n:n + ne]).all()
                hq_ref = np.zeros((cap_e, wl.F // 32, 36), np.uint8)
                orc.swiglu_q8_1(np.nan_to_num(ref).astype(np.float32), wl.F, n, n + ne, hq_ref)
                flips, scale_diffs = H.q8_1_code_flips(hq[n:n + ne], hq_ref[n:n + ne])
                # ... and down to the scattered rows (fp64), from the oracle's h
                oref = np.full((n + 6, wl.N), np.nan)
                orc.grouped_gemv(L.dn_t, wl.F, wl.N, dnb, ge[:1], gs[:2], 1, hq_ref, ent_out=ed, out=oref,
                                 cb=L.cb_dn)
                rows = sorted(own_out)
                bound = TOL if flips == 0 and scale_diffs == 0 else 2e-3
                assert H.rel_err(out[rows], oref[rows]) <= bound, (gg, ne, flips)
                # the GPU's down on its own h against the oracle's down on the same h: 1e-5
                oref_own = np.full((n + 6, wl.N), np.nan)
                orc.grouped_gemv(L.dn_t, wl.F, wl.N, dnb, ge[:1], gs[:2], 1, hq, ent_out=ed, out=oref_own,
                                 cb=L.cb_dn)
                assert H.rel_err(out[rows], oref_own[rows]) <= TOL, (gg, ne)


def test_device_errors_are_reported_and_skipped(m, orc):
    wl = synth.WORKLOADS["tiny"]
    L = H.make_layer(wl, (synth.Q8_0, synth.Q8_0), 1)
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    G = int(B.n_groups.item())
    # n_groups above cap: clamped, reported
    B.n_groups.fill_(B.cap_groups + 5)
    H.expert_call(m, L, B)()
    torch.cuda.synchronize()
    assert int(B.err.item()) & 1
    # an expert id out of range: that group skipped and reported, the other written
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    ge = B.grp_expert.cpu().numpy(); gs = B.grp_start.cpu().numpy()
    B.grp_expert[0] = wl.E + 3
    H.expert_call(m, L, B)()
    torch.cuda.synchronize()
    assert int(B.err.item()) & 2
    gu = B.gu.cpu().numpy()
    assert np.isnan(gu[gs[0]:gs[1]]).all() and not np.isnan(gu[gs[1]:gs[G]]).any()
