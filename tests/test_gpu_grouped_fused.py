"""The one-launch grouped call (moe_expert_grouped_fused) against the three-launch one
(moe_expert_grouped) and the CPU oracle.

#363 "experts: smaller and fewer launches for the verify window's PCIe call" ("What changes",
"Exactness") fixes the call's contract: groups and a device-side n_groups come from the caller,
entries may start past 0, destinations are scattered and rows outside the call stay untouched. The
fused launch performs the same arithmetic in the same order, so every row it writes must equal the
three-launch call's bit for bit; rows it does not own stay NaN.
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


def _bits(t):
    return t.view(torch.int32).cpu().numpy()


def _sync(m, B, wl, pair=False):
    n = m.grouped_fused_sync_ints(B.cap_groups, B.cap_entries, wl.F)
    return torch.zeros((2 if pair else 1) * n, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("wname,pair,T,xt", [("verify", (synth.CB2, synth.NL4), 4, None),
                                             ("verify", (synth.CB2, synth.NL4), 4, synth.CB2X),
                                             ("tiny", (synth.Q8_0, synth.Q8_0), 1, None),
                                             ("sweep", (synth.CB3, synth.Q8_0), 4, None)])
def test_fused_equals_three_launch_call(m, orc, wname, pair, T, xt):
    wl = synth.WORKLOADS[wname]
    L0 = H.make_layer(wl, pair, T)
    L = H.transcoded(m, L0, xt) if xt else L0
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    H.expert_call(m, L, B)()
    torch.cuda.synchronize()
    ref = (B.gu.clone(), B.hq.clone(), B.out.clone())
    for r in range(2):  # two calls in a row on one sync array
        B.gu.fill_(float("nan")); B.out.fill_(float("nan")); B.hq.fill_(0xA5)
        sync = _sync(m, B, wl) if r == 0 else sync
        H.expert_call(m, L, B).call_fused(sync)
        torch.cuda.synchronize()
        assert int(B.err.item()) == 0
        assert np.array_equal(_bits(B.gu), _bits(ref[0]))
        assert torch.equal(B.hq, ref[1])
        assert np.array_equal(_bits(B.out), _bits(ref[2]))
        assert tuple(sync[:3].tolist()) == (0, 0, r + 1)
    # and against the oracle's chain
    o = H.oracle_call(orc, L0)
    flips, scale_diffs = H.q8_1_code_flips(B.hq.cpu().numpy(), o["hq"])
    err = H.rel_err(B.out.cpu().numpy(), o["out"])
    assert err <= (TOL if flips == 0 and scale_diffs == 0 else 2e-3), (err, flips)


def test_fused_second_call(m, orc):
    """The layer's second (PCIe) call: n_groups in {0, 1}, 1-2 entries numbered after the first
    call's 32, scattered destinations; equal to the three-launch call bit for bit, rows it does not
    own untouched, and the owned out rows against the oracle's chain."""
    wl = synth.WORKLOADS["sparse"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    n = L.T * wl.k
    xq = orc.quantize_q8_1(L.x)
    gub = H.host_blobs(L, [17], "gu")
    dnb = H.host_blobs(L, [17], "dn")
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
        H.expert_call(m, L, B)()
        torch.cuda.synchronize()
        ref = (B.gu.clone(), B.hq.clone(), B.out.clone())
        sync = _sync(m, B, wl)
        B.gu.fill_(float("nan")); B.out.fill_(float("nan")); B.hq.fill_(0xA5)
        H.expert_call(m, L, B).call_fused(sync)
        torch.cuda.synchronize()
        assert int(B.err.item()) == 0
        assert np.array_equal(_bits(B.gu), _bits(ref[0]))
        assert torch.equal(B.hq, ref[1])
        assert np.array_equal(_bits(B.out), _bits(ref[2]))
        out = B.out.cpu().numpy()
        own_out = set(ed[n:n + ne].tolist()) if ng else set()
        for i in range(n + 6):
            assert np.isnan(out[i]).all() == (i not in own_out)
        if ng:
            gu_ref = np.full((cap_e, 2 * wl.F), np.nan)
            orc.grouped_gemv(L.gu_t, wl.N, 2 * wl.F, gub, ge[:1], gs[:2], 1, xq, ent_in=es, out=gu_ref, cb=L.cb_gu)
            hq_ref = np.zeros((cap_e, wl.F // 32, 36), np.uint8)
            orc.swiglu_q8_1(np.nan_to_num(gu_ref).astype(np.float32), wl.F, n, n + ne, hq_ref)
            flips, scale_diffs = H.q8_1_code_flips(B.hq.cpu().numpy()[n:n + ne], hq_ref[n:n + ne])
            oref = np.full((n + 6, wl.N), np.nan)
            orc.grouped_gemv(L.dn_t, wl.F, wl.N, dnb, ge[:1], gs[:2], 1, hq_ref, ent_out=ed, out=oref, cb=L.cb_dn)
            rows = sorted(own_out)
            assert H.rel_err(out[rows], oref[rows]) <= (TOL if flips == 0 and scale_diffs == 0 else 2e-3)


def test_fused_sync_pair_alternating(m, orc):
    """Four calls alternating the halves of one sync pair: each equals its three-launch call."""
    wl = synth.WORKLOADS["verify"]
    Ls = [H.make_layer(wl, (synth.CB2, synth.NL4), 4, layer=l) for l in range(4)]
    Bs = [H.make_bufs(L) for L in Ls]
    refs = []
    for L, B in zip(Ls, Bs):
        H.gpu_route_and_quantize(m, L, B)
        H.expert_call(m, L, B)()
        torch.cuda.synchronize()
        refs.append(B.out.clone())
    sync = _sync(m, Bs[0], wl, pair=True)
    for i, (L, B) in enumerate(zip(Ls, Bs)):
        B.out.fill_(float("nan"))
        c = H.expert_call(m, L, B, flags=m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if i % 2 else 0))
        c.call_fused(sync)
    torch.cuda.synchronize()
    for B, r in zip(Bs, refs):
        assert int(B.err.item()) == 0
        assert np.array_equal(_bits(B.out), _bits(r))


def test_fused_empty_calls_in_a_sync_pair(m, orc):
    """Empty calls (n_groups 0, which end right after the dependency wait) between real calls on
    alternating halves of one sync pair: each real call equals its three-launch call, the empty
    calls write nothing, and every counter is zero again at the end."""
    wl = synth.WORKLOADS["verify"]
    Ls = [H.make_layer(wl, (synth.CB2, synth.NL4), 4, layer=l) for l in range(4)]
    Bs = [H.make_bufs(L) for L in Ls]
    refs = []
    for L, B in zip(Ls, Bs):
        H.gpu_route_and_quantize(m, L, B)
        H.expert_call(m, L, B)()
        torch.cuda.synchronize()
        refs.append(B.out.clone())
    E0 = H.make_bufs(Ls[0])
    E0.grp_expert.copy_(Bs[0].grp_expert); E0.grp_start.copy_(Bs[0].grp_start)
    E0.ent_src.copy_(Bs[0].ent_src); E0.ent_dst.copy_(Bs[0].ent_dst); E0.xq.copy_(Bs[0].xq)
    E0.n_groups.fill_(0)
    sync = _sync(m, Bs[0], wl, pair=True)
    # halves: L0 even, empty odd, L1 even, empty odd, L2 even, L3 odd
    seq = [(Ls[0], Bs[0]), (Ls[0], E0), (Ls[1], Bs[1]), (Ls[0], E0), (Ls[2], Bs[2]), (Ls[3], Bs[3])]
    for B in Bs:
        B.out.fill_(float("nan"))
    for i, (L, B) in enumerate(seq):
        c = H.expert_call(m, L, B, flags=m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if i % 2 else 0))
        c.call_fused(sync)
    torch.cuda.synchronize()
    for B, r in zip(Bs, refs):
        assert int(B.err.item()) == 0
        assert np.array_equal(_bits(B.out), _bits(r))
    assert int(E0.err.item()) == 0
    assert torch.isnan(E0.out).all() and torch.isnan(E0.gu).all()
    # the last call (odd half) reset the even half; its own counters are zeroed by the next call,
    # and its exit count is not used in pair mode
    half = sync.numel() // 2
    s = sync.cpu().numpy()
    assert s[0] == 0 and s[1] == 0
    assert s[half] == 0


def test_fused_bad_groups_are_reported_and_skipped(m, orc):
    """n_groups above cap is clamped (MOE_ERR_NGROUPS); a group with an expert id out of range
    (MOE_ERR_EXPERT) or an entry whose source or destination row is out of range (MOE_ERR_ENTRY)
    is skipped and its rows stay NaN; every other group equals the three-launch call. (The CTAs
    whose first work item is a unit of a skipped group copy nothing ahead of the tables.)"""
    wl = synth.WORKLOADS["verify"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    H.expert_call(m, L, B)()
    torch.cuda.synchronize()
    ref = B.out.clone()
    gs = B.grp_start.cpu().numpy()
    G = int(B.n_groups.item())
    ed = B.ent_dst.cpu().numpy()
    # group 0: expert out of range; group 1: one entry's source row out of range; group 2: one
    # entry's destination row out of range
    assert G >= 4
    B.grp_expert[0] = wl.E + 5
    B.ent_src[int(gs[1])] = 99
    B.ent_dst[int(gs[3]) - 1] = B.out.shape[0] + 1
    B.out.fill_(float("nan"))
    sync = _sync(m, B, wl)
    H.expert_call(m, L, B).call_fused(sync)
    torch.cuda.synchronize()
    assert int(B.err.item()) == 2 | 8
    out, r = B.out.cpu().numpy(), ref.cpu().numpy()
    skipped = set(range(gs[0], gs[3]))
    for e in range(gs[0], gs[G]):
        row = int(ed[e])
        if e in skipped:
            assert np.isnan(out[row]).all()
        else:
            assert np.array_equal(out[row].view(np.int32), r[row].view(np.int32))
    # n_groups above cap: clamped to cap (the slots past G hold nothing: zero-entry groups)
    B2 = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B2)
    B2.n_groups.fill_(B2.cap_groups + 3)
    H.expert_call(m, L, B2).call_fused(_sync(m, B2, wl))
    torch.cuda.synchronize()
    assert int(B2.err.item()) & 1


def test_staged_host_expert_call(m, orc):
    """The residency split: a second call whose expert lives in pinned host memory, copied into a
    device staging slot with moe_stage_blobs (its copy kernel, pinned blobs) and run with the
    one-launch call, first eagerly and then captured with the copies in one CUDA graph; its out
    rows equal the same call on the device-resident copy of the expert bit for bit, and the
    oracle's chain."""
    wl = synth.WORKLOADS["sparse"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    n = L.T * wl.k
    x = 23
    gub = H.host_blobs(L, [x], "gu")
    dnb = H.host_blobs(L, [x], "dn")
    host = [torch.from_numpy(gub[x]).pin_memory(), torch.from_numpy(dnb[x]).pin_memory()]
    slots = [torch.empty(h.numel() + 64, dtype=torch.uint8, device="cuda") for h in host]
    cap_e = n + 2
    B = H.make_bufs(L, cap_entries=cap_e, out_rows=n + 6)
    m.quantize_q8_1(torch.from_numpy(L.x).cuda(), B.xq)
    ge = np.array([x] + [0] * (n - 1), np.int32)
    gs = np.array([n, n + 2] + [0] * (n - 1), np.int32)
    es = np.full(cap_e, -7, np.int32); es[n:n + 2] = [3, 1]
    ed = np.full(cap_e, -7, np.int32); ed[n:n + 2] = [n + 4, 2]
    B.grp_expert.copy_(torch.from_numpy(ge)); B.grp_start.copy_(torch.from_numpy(gs)); B.n_groups.fill_(1)
    B.ent_src.copy_(torch.from_numpy(es)); B.ent_dst.copy_(torch.from_numpy(ed))
    # reference: the same call on the device-resident pool
    sync = _sync(m, B, wl)
    H.expert_call(m, L, B).call_fused(sync)
    torch.cuda.synchronize()
    ref = B.out.clone()
    # staged: pointer tables whose entry x names the slots
    tab_gu, tab_dn = L.tab_gu.clone(), L.tab_dn.clone()
    tab_gu[x] = slots[0].data_ptr()
    tab_dn[x] = slots[1].data_ptr()
    Ls = H.Layer(**{**L.__dict__, "tab_gu": tab_gu, "tab_dn": tab_dn})
    for s_ in slots:
        s_.fill_(0x5A)
    B.out.fill_(float("nan"))
    m.stage_blobs(host, slots)
    H.expert_call(m, Ls, B).call_fused(sync)
    torch.cuda.synchronize()
    assert int(B.err.item()) == 0
    assert np.array_equal(_bits(B.out), _bits(ref))
    # the copies and the call captured together in one graph, replayed twice
    for s_ in slots:
        s_.fill_(0x5A)
    st = torch.cuda.Stream()
    call = H.expert_call(m, Ls, B)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st, capture_error_mode="relaxed"):
        m.stage_blobs(host, slots)
        call.call_fused(sync)
    for _ in range(2):
        B.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_bits(B.out), _bits(ref))
    # the oracle on the host blobs
    xq = orc.quantize_q8_1(L.x)
    gu_ref = np.full((cap_e, 2 * wl.F), np.nan)
    orc.grouped_gemv(L.gu_t, wl.N, 2 * wl.F, gub, ge[:1], gs[:2], 1, xq, ent_in=es, out=gu_ref, cb=L.cb_gu)
    hq_ref = np.zeros((cap_e, wl.F // 32, 36), np.uint8)
    orc.swiglu_q8_1(np.nan_to_num(gu_ref).astype(np.float32), wl.F, n, n + 2, hq_ref)
    flips, scale_diffs = H.q8_1_code_flips(B.hq.cpu().numpy()[n:n + 2], hq_ref[n:n + 2])
    oref = np.full((n + 6, wl.N), np.nan)
    orc.grouped_gemv(L.dn_t, wl.F, wl.N, dnb, ge[:1], gs[:2], 1, hq_ref, ent_out=ed, out=oref, cb=L.cb_dn)
    rows = [2, n + 4]
    assert H.rel_err(B.out.cpu().numpy()[rows], oref[rows]) <= (TOL if flips == 0 and scale_diffs == 0 else 2e-3)


def test_stage_blobs_kernel_and_copy_paths(m):
    """moe_stage_blobs: pinned 16-byte aligned blobs of whole 16-byte words go through the copy
    kernel (ten of them: two launches of at most eight), a pinned blob of an odd size and pageable
    blobs through cudaMemcpyAsync; every slot ends equal to its source byte for byte, eagerly and,
    for the pinned blobs, captured in a CUDA graph."""
    g = torch.Generator().manual_seed(5)
    sizes = [1_105_920, 2_088_960] + [4096 * (i + 1) + 16 * i for i in range(8)]
    pinned = [torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory() for n in sizes]
    odd = torch.randint(0, 256, (1000,), dtype=torch.uint8, generator=g).pin_memory()
    pageable = [torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g) for n in (65536, 4112)]
    srcs = pinned + [odd] + pageable
    slots = [torch.zeros(h.numel(), dtype=torch.uint8, device="cuda") for h in srcs]
    m.stage_blobs(srcs, slots)
    torch.cuda.synchronize()
    for h, d in zip(srcs, slots):
        assert torch.equal(d.cpu(), h)
    for d in slots:
        d.zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        m.stage_blobs(pinned + [odd], slots[:len(pinned) + 1], stream=s)
    graph.replay()
    torch.cuda.synchronize()
    for h, d in zip(pinned + [odd], slots):
        assert torch.equal(d.cpu(), h)
