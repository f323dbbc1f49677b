"""The fused layer call (moe_expert_layer: routing, q8_1, gate/up, SwiGLU + q8_1 and down in one
launch) against the separate steps and against the CPU oracle.

The fused call performs the same arithmetic in the same order as the separate kernels, so every
output (grouping, activation q8_1, gate/up rows, q8_1 h rows, output rows) must match them bit for
bit; the output is also checked against the oracle directly (max|err| / max|ref| <= 1e-5 unless
an h code flipped, as in the end-to-end parity test).
"""
import numpy as np
import pytest
import torch

import harness as H
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-5

CASES = [("tiny", (synth.Q8_0, synth.Q8_0), 1, None), ("verify", (synth.CB2, synth.NL4), 4, None),
         ("window48", (synth.CB3, synth.NL4), 1, None), ("window48", (synth.CB3, synth.NL4), 2, synth.CB3X),
         ("window48", (synth.CB3, synth.NL4), 4, synth.CB3X), ("verify", (synth.CB2, synth.NL4), 4, synth.CB2X),
         ("verify", (synth.CB2, synth.NL4), 8, None), ("window48", (synth.CB3, synth.NL4), 6, synth.CB3X),
         ("sweep", (synth.Q4B, synth.NL4), 4, None), ("sweep", (synth.CB3, synth.Q8_0), 4, None),
         ("sweep", (synth.Q8_0, synth.Q8_0), 4, None), ("sweep", (synth.CB2, synth.NL4), 4, None),
         ("sweep", (synth.Q4B, synth.Q8_0), 4, None), ("sweep", (synth.CB3, synth.NL4), 4, None),
         ("sweep", (synth.Q8_0, synth.NL4), 4, None), ("sweep", (synth.CB2, synth.Q8_0), 4, None)]
CASE_IDS = [f"{c[0]}-{synth.NAMES[c[1][0]]}-{synth.NAMES[c[1][1]]}-T{c[2]}" + (f"-{synth.NAMES[c[3]]}" if c[3] else "")
            for c in CASES]


def _left_clean(sync, calls):
    """The control words a call leaves: exit and work counters zero, the epoch advanced once per
    call (the flagged h copies after them keep the last call's flag)."""
    exit_, work, epoch = (int(v) for v in sync[:3].tolist())
    assert (exit_, work, epoch) == (0, 0, calls)


@pytest.fixture(scope="module")
def m():
    import quantized_routed_expert_grouped_gb300 as mod
    mod.lib()
    return mod


class Fused:
    """Device buffers of one fused call (NaN / 0xA5 prefilled so unwritten rows show)."""

    def __init__(self, m, L, ids=None, flags=1):
        wl, T = L.wl, L.T
        n = T * wl.k
        dev = "cuda"
        i32 = dict(dtype=torch.int32, device=dev)
        self.ids = torch.from_numpy(L.ids if ids is None else ids).to(dev)
        self.x = torch.from_numpy(L.x).to(dev)
        self.out = torch.full((n, wl.N), float("nan"), dtype=torch.float32, device=dev)
        self.gu = torch.full((n, 2 * wl.F), float("nan"), dtype=torch.float32, device=dev)
        self.hq = torch.full((n, wl.F // 32, 36), 0xA5, dtype=torch.uint8, device=dev)
        self.sync = torch.zeros(m.layer_sync_ints(T, wl.k, wl.F), **i32)
        self.ge = torch.full((n,), -7, **i32)
        self.gs = torch.full((n + 1,), -7, **i32)
        self.ng = torch.full((1,), -7, **i32)
        self.es = torch.full((n,), -7, **i32)
        self.ed = torch.full((n,), -7, **i32)
        self.xq = torch.full((T, wl.N // 32, 36), 0xA5, dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, **i32)
        self.call = m.LayerCall(L.gu_t, L.cb_gu_d, L.dn_t, L.cb_dn_d, wl.N, wl.F, L.tab_gu, L.tab_dn, wl.E, self.ids,
                                self.x, self.out, self.gu, self.hq, self.sync, self.err, flags, self.ge, self.gs,
                                self.ng, self.es, self.ed, self.xq)


def _separate(m, L):
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    H.expert_call(m, L, B)()
    torch.cuda.synchronize()
    return B


def _bits(t):
    return t.view(torch.int32).cpu().numpy()


def _same_as_separate(F, B, ntot):
    G = int(B.n_groups.item())
    assert int(F.ng.item()) == G
    assert torch.equal(F.ge[:G], B.grp_expert[:G]) and torch.equal(F.gs[:G + 1], B.grp_start[:G + 1])
    assert torch.equal(F.es[:ntot], B.ent_src[:ntot]) and torch.equal(F.ed[:ntot], B.ent_dst[:ntot])
    assert torch.equal(F.xq, B.xq)
    assert np.array_equal(_bits(F.gu[:ntot]), _bits(B.gu[:ntot]))
    assert torch.equal(F.hq[:ntot], B.hq[:ntot])
    assert np.array_equal(_bits(F.out), _bits(B.out))


@pytest.mark.parametrize("wname,pair,T,xt", CASES, ids=CASE_IDS)
def test_layer_equals_separate_steps_and_oracle(m, orc, wname, pair, T, xt):
    _check_layer(m, orc, synth.WORKLOADS[wname], pair, T, xt)


# The fused call at its entry capacity (T*k = 512) on small shapes: 64 tokens, top-8 of 64
# experts, so about eight entries per group (four batches of two each), CB3 gate/up read directly
# (its codebook staged in shared memory) and NL4 down.
CAP = synth.Workload("cap512", 1, (64,), 64, 8, 512, 256, ((synth.CB3, synth.NL4),), seed=66)


def test_layer_at_entry_capacity(m, orc):
    _check_layer(m, orc, CAP, CAP.pairs[0], 64, None)


# Degenerate shapes: one expert (every token's only id: one group of T entries, two batches),
# two experts with top-2 (two groups of T entries each, an odd batch), the smallest layer
# (n_embd = n_ff = 256, one chunk per row).
DEGENERATE = [synth.Workload("one_expert", 1, (4,), 1, 1, 256, 256, ((synth.Q8_0, synth.NL4),), seed=71),
              synth.Workload("two_experts", 1, (3,), 2, 2, 512, 256, ((synth.CB2, synth.Q8_0),), seed=72),
              synth.Workload("min_shape", 1, (1,), 4, 2, 256, 256, ((synth.CB3, synth.NL4),), seed=73)]


@pytest.mark.parametrize("wl", DEGENERATE, ids=[w.name for w in DEGENERATE])
def test_layer_degenerate_shapes(m, orc, wl):
    _check_layer(m, orc, wl, wl.pairs[0], wl.T[0], None)


def _check_layer(m, orc, wl, pair, T, xt):
    L0 = H.make_layer(wl, pair, T)
    L = H.transcoded(m, L0, xt) if xt else L0
    n = T * wl.k
    B = _separate(m, L)
    F = Fused(m, L)
    F.call()
    torch.cuda.synchronize()
    assert int(F.err.item()) == 0 and int(B.err.item()) == 0
    _same_as_separate(F, B, n)
    _left_clean(F.sync, 1)
    ref = H.oracle_call(orc, L0)
    flips, scale_diffs = H.q8_1_code_flips(F.hq.cpu().numpy(), ref["hq"])
    assert flips <= max(2, n * wl.F // 4096) and scale_diffs <= 2, (flips, scale_diffs)
    err = H.rel_err(F.out.cpu().numpy(), ref["out"])
    assert err <= (TOL if flips == 0 and scale_diffs == 0 else 2e-3), (err, flips)
    assert H.rel_err(F.gu.cpu().numpy(), ref["gu"]) <= TOL


def test_layer_repeated_calls_pdl_and_graph(m, orc):
    """Several layers sharing one sync array, eager (with and without PDL) and captured in a CUDA
    graph replayed twice: identical outputs every time, counters left zero and the epoch advanced
    once per call (18 calls)."""
    wl = synth.WORKLOADS["window48"]
    layers = [H.transcoded(m, H.make_layer(wl, (synth.CB3, synth.NL4), 3, layer=l), synth.CB3X) for l in range(3)]
    fs = [Fused(m, L) for L in layers]
    sync = fs[0].sync
    for f in fs:  # one shared counter array
        f.call.c.sync = sync.data_ptr()
    for f in fs:
        f.call()
    torch.cuda.synchronize()
    base = [f.out.clone() for f in fs]
    for L, f in zip(layers, fs):
        _same_as_separate(f, _separate(m, L), L.T * wl.k)
    for flags in (0, 1):
        for f in fs:
            f.call.c.flags = flags
            f.out.fill_(float("nan"))
            f.call()
        torch.cuda.synchronize()
        for f, b in zip(fs, base):
            assert torch.equal(f.out.view(torch.int32), b.view(torch.int32))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in fs:
            f.call(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for f in fs:
            f.call()
    for _ in range(2):
        for f in fs:
            f.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for f, b in zip(fs, base):
            assert torch.equal(f.out.view(torch.int32), b.view(torch.int32))
    assert all(int(f.err.item()) == 0 for f in fs)
    _left_clean(sync, 18)


def test_layer_sync_pair_alternating_halves(m, orc):
    """MOE_F_SYNC_PAIR: four layers at T = 4 alternate the two halves of one sync array (each call
    resets the other half instead of its last CTA resetting its own), eager with PDL and in a CUDA
    graph replayed twice: the outputs equal the default mode's bit for bit, and after every call
    the half the next call uses has zero counters and its epoch advanced once per reset."""
    wl = synth.WORKLOADS["window48"]
    layers = [H.transcoded(m, H.make_layer(wl, (synth.CB3, synth.NL4), 4, layer=l), synth.CB3X) for l in range(4)]
    base = []
    for L in layers:  # default mode, each with its own counters
        f = Fused(m, L)
        f.call()
        torch.cuda.synchronize()
        assert int(f.err.item()) == 0
        base.append(f.out.clone())
    half = m.layer_sync_ints(4, wl.k, wl.F)
    pair = torch.zeros(2 * half, dtype=torch.int32, device="cuda")
    fs = [Fused(m, L) for L in layers]
    for i, f in enumerate(fs):
        f.call.c.sync = pair.data_ptr()
        f.call.c.flags = m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if i % 2 else 0)
    for i, f in enumerate(fs):  # one at a time: the next call's half is reset after each
        f.call()
        torch.cuda.synchronize()
        nxt = pair[half:] if i % 2 == 0 else pair[:half]
        _left_clean(nxt, i // 2 + 1)
    for f, b in zip(fs, base):
        assert int(f.err.item()) == 0
        assert torch.equal(f.out.view(torch.int32), b.view(torch.int32))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for f in fs:
            f.call()
    for r in range(2):
        for f in fs:
            f.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for f, b in zip(fs, base):
            assert torch.equal(f.out.view(torch.int32), b.view(torch.int32))
        _left_clean(pair[:half], 4 + 2 * r)  # reset by every odd call: two per pass
    assert all(int(f.err.item()) == 0 for f in fs)


def _window_layers(m, wl, T, layers):
    return [H.transcoded(m, H.make_layer(wl, (synth.CB3, synth.NL4), T, layer=l), synth.CB3X) for l in layers]


def test_layer_epoch_wrap(m, orc):
    """The call epoch skips 2^32 - 1 (whose flag would be 0, the flag of a pair never written): the
    call that would reach it zeroes every h pair a call on the array has used (word 3) and
    restarts the epoch at 0. One array sized for T = 4 serves a T = 4 call (its pairs carry flag
    1), then, with the epoch set just below the wrap, a T = 2 call that wraps it, then a T = 4 call
    whose flag is 1 again. Without the clearing, that last call's down phase would take the first
    call's stale h blocks of entries 16..31 (another layer's data) as its own."""
    wl = synth.WORKLOADS["window48"]
    LA, = _window_layers(m, wl, 4, [1])
    LB, = _window_layers(m, wl, 2, [2])
    LC, = _window_layers(m, wl, 4, [3])
    refB, refC = _separate(m, LB), _separate(m, LC)
    ext = 4 * wl.k * 9 * (wl.F // 32)
    sync = torch.zeros(m.layer_sync_ints(4, wl.k, wl.F), dtype=torch.int32, device="cuda")
    fs = [Fused(m, L) for L in (LA, LB, LC)]
    for f in fs:
        f.call.c.sync = sync.data_ptr()
    fs[0].call()
    torch.cuda.synchronize()
    assert tuple(sync[:4].tolist()) == (0, 0, 1, ext)
    sync[2] = -2  # epoch 2^32 - 2: the next call's flag is 2^32 - 1
    fs[1].call()
    torch.cuda.synchronize()
    assert tuple(sync[:4].tolist()) == (0, 0, 0, ext)  # wrapped: epoch 0 again
    assert not sync[4:].any()  # every pair used so far zeroed
    assert np.array_equal(_bits(fs[1].out), _bits(refB.out))
    fs[2].call()
    torch.cuda.synchronize()
    assert all(int(f.err.item()) == 0 for f in fs)
    assert np.array_equal(_bits(fs[2].out), _bits(refC.out))
    _same_as_separate(fs[2], refC, 4 * wl.k)
    assert tuple(sync[:4].tolist()) == (0, 0, 1, ext)


def test_layer_epoch_wrap_sync_pair(m, orc):
    """The same with MOE_F_SYNC_PAIR, where a call advances the other half's epoch on its way out:
    call 0 (first half, flag 1), the first half's epoch set just below the wrap, call 1 (second
    half) wraps the first half and clears its pairs, call 2 (first half, flag 1 again) must not
    take call 0's stale h blocks."""
    wl = synth.WORKLOADS["window48"]
    Ls = _window_layers(m, wl, 4, [4, 5, 6])
    refs = [_separate(m, L) for L in Ls]
    half = m.layer_sync_ints(4, wl.k, wl.F)
    ext = 4 * wl.k * 9 * (wl.F // 32)
    pair = torch.zeros(2 * half, dtype=torch.int32, device="cuda")
    fs = [Fused(m, L) for L in Ls]
    for i, f in enumerate(fs):
        f.call.c.sync = pair.data_ptr()
        f.call.c.flags = m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if i % 2 else 0)
    fs[0].call()
    torch.cuda.synchronize()
    # the first half keeps its counters until call 1 resets it; its extent is recorded
    assert tuple(pair[2:4].tolist()) == (0, ext) and tuple(pair[half:half + 3].tolist()) == (0, 0, 1)
    pair[2] = -2
    fs[1].call()
    torch.cuda.synchronize()
    assert tuple(pair[:4].tolist()) == (0, 0, 0, ext) and not pair[4:half].any()
    fs[2].call()
    torch.cuda.synchronize()
    for f, r in zip(fs, refs):
        assert int(f.err.item()) == 0
        assert np.array_equal(_bits(f.out), _bits(r.out))


def test_layer_timeout_path(m, orc):
    """The abort path of the fused kernel, made to run by MOE_F_TEST_EXPIRE: every CTA's down
    staging waits for a flag that no call writes, gives up after the wait limit (~1 s), sets
    MOE_ERR_TIMEOUT, stops its producer, lets its consumers drain and waits for its own copies in
    flight. The call ends (no hang) and the context stays usable: with the sync array zeroed
    again, the next call equals the separate path bit for bit."""
    import time
    wl = synth.WORKLOADS["verify"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    n = L.T * wl.k
    B = _separate(m, L)
    F = Fused(m, L)
    F.call.c.flags = m.F_TEST_EXPIRE
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    F.call()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(F.err.item()) & 64, int(F.err.item())  # MOE_ERR_TIMEOUT
    assert 0.5 < dt < 30, dt
    assert np.isnan(F.out.cpu().numpy()).all()  # no down row was written
    F.sync.zero_()
    F.err.zero_()
    F.out.fill_(float("nan"))
    F.call.c.flags = m.F_PDL
    F.call()
    torch.cuda.synchronize()
    assert int(F.err.item()) == 0
    _same_as_separate(F, B, n)
    _left_clean(F.sync, 1)


def test_layer_dropped_ids_and_empty(m, orc):
    wl = synth.WORKLOADS["verify"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    ids = L.ids.copy()
    ids[0, 3] = -1
    ids[2, 0] = wl.E
    ids[3, 7] = 10 ** 6
    F = Fused(m, L, ids=ids)
    F.call()
    torch.cuda.synchronize()
    assert int(F.err.item()) == 128  # MOE_ERR_ROUTE only
    _left_clean(F.sync, 1)
    # the separate path on the same ids
    Ld = H.Layer(**{**L.__dict__, "ids": ids})
    B = _separate(m, Ld)
    ntot = int(B.grp_start[int(B.n_groups.item())].item())
    assert ntot == wl.k * L.T - 3
    _same_as_separate(F, B, ntot)
    out = F.out.cpu().numpy()
    for r in (0 * wl.k + 3, 2 * wl.k + 0, 3 * wl.k + 7):
        assert np.isnan(out[r]).all()
    # every id dropped: nothing computed, nothing written
    F2 = Fused(m, L, ids=np.full_like(L.ids, -1))
    F2.call()
    torch.cuda.synchronize()
    assert int(F2.err.item()) == 128 and int(F2.ng.item()) == 0
    assert torch.isnan(F2.out).all() and torch.isnan(F2.gu).all() and (F2.hq == 0xA5).all()
    _left_clean(F2.sync, 1)
    assert not F2.sync[4:].any()  # no h block written


def test_layer_misaligned_expert_is_skipped(m, orc):
    """A weight pointer that is not 16-byte aligned: that group is skipped with MOE_ERR_ALIGN, no
    wait times out, and every other entry's output equals the separate path's."""
    wl = synth.WORKLOADS["verify"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4)
    bad = int(L.ids[1, 2])
    B = _separate(m, L)
    tab = L.tab_gu.clone()
    tab[bad] += 2
    Lb = H.Layer(**{**L.__dict__, "tab_gu": tab})
    F = Fused(m, Lb)
    F.call()
    torch.cuda.synchronize()
    assert int(F.err.item()) == 16
    _left_clean(F.sync, 1)
    out, ref = F.out.cpu().numpy(), B.out.cpu().numpy()
    for t in range(L.T):
        for s in range(wl.k):
            r = t * wl.k + s
            if int(L.ids[t, s]) == bad:
                assert np.isnan(out[r]).all()
            else:
                assert np.array_equal(out[r].view(np.int32), ref[r].view(np.int32))


@pytest.mark.parametrize("layer", [17, 47])
def test_layer_sampled_window_layers(m, orc, layer):
    """Other layers of the 48-layer window (their own experts, routing and activations) at T = 4 on
    the slot layout: fused equals separate bit for bit and matches the oracle."""
    wl = synth.WORKLOADS["window48"]
    L0 = H.make_layer(wl, (synth.CB3, synth.NL4), 4, layer=layer)
    L = H.transcoded(m, L0, synth.CB3X)
    B = _separate(m, L)
    F = Fused(m, L)
    F.call()
    torch.cuda.synchronize()
    assert int(F.err.item()) == 0
    _same_as_separate(F, B, 4 * wl.k)
    ref = H.oracle_call(orc, L0)
    flips, scale_diffs = H.q8_1_code_flips(F.hq.cpu().numpy(), ref["hq"])
    err = H.rel_err(F.out.cpu().numpy(), ref["out"])
    assert err <= (TOL if flips == 0 and scale_diffs == 0 else 2e-3), (err, flips)

