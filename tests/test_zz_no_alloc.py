"""The allocation-free expert call, moe_expert_grouped_static, through the C ABI.

It is for callers that cannot allocate device memory for a call's scratch (an engine that
reserves all device memory at start-up, a plugin whose host framework owns every allocation, a
latency-critical path that cannot take cudaMalloc's implicit synchronisation): it keeps the
gate/up and q8_1 h scratch in a static device buffer inside the library. Its output must match
moe_expert_grouped (caller-provided scratch) within the parity tolerance, on two calls in a row.
This file sorts last so that a stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

import harness as H
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-5


def _run(m, L, B, static, dst=None):
    B.out.fill_(float("nan"))
    call = H.expert_call(m, L, B)
    if static:
        call.call_static()
    else:
        call()
    torch.cuda.synchronize()
    if dst is None:
        return B.out.clone()
    dst.copy_(B.out)
    torch.cuda.synchronize()
    return dst


def _same_bits(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_static_scratch_call_matches_allocating_call():
    import quantized_routed_expert_grouped_gb300 as m
    m.lib()
    for wname, pair, T in (("verify", (synth.CB2, synth.NL4), 4), ("tiny", (synth.Q8_0, synth.Q8_0), 1)):
        wl = synth.WORKLOADS[wname]
        L = H.make_layer(wl, pair, T)
        B = H.make_bufs(L)
        H.gpu_route_and_quantize(m, L, B)
        ref = _run(m, L, B, static=False)
        assert not torch.isnan(ref).any()
        got = torch.empty_like(ref)
        # the first static call on a device may load the library's static buffer (the module is
        # loaded lazily: its 4 MiB appear then, once, and stay until exit); it is checked too
        _run(m, L, B, static=True, dst=got)
        assert _same_bits(got, ref)
        torch.cuda.synchronize()
        free0, allocated0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        for _ in range(2):  # two calls in a row share (and reuse) the static buffer
            _run(m, L, B, static=True, dst=got)
            assert int(B.err.item()) == 0
            # the same kernels on the same inputs, only the scratch lives elsewhere: the same
            # bits (which is within any tolerance)
            assert H.rel_err(got.cpu().numpy(), ref.cpu().numpy()) <= TOL
            assert _same_bits(got, ref)
        # and the calls allocated no device memory
        assert torch.cuda.memory_allocated() == allocated0
        assert torch.cuda.mem_get_info()[0] >= free0
    # a second routing after the first: stale scratch from the previous call must not leak
    wl = synth.WORKLOADS["verify"]
    L2 = H.make_layer(wl, (synth.CB2, synth.NL4), 4, layer=1)
    B2 = H.make_bufs(L2)
    H.gpu_route_and_quantize(m, L2, B2)
    ref2 = _run(m, L2, B2, static=False)
    got2 = _run(m, L2, B2, static=True)
    assert H.rel_err(got2.cpu().numpy(), ref2.cpu().numpy()) <= TOL
    assert _same_bits(got2, ref2)


def test_static_scratch_rejects_oversize_calls():
    import quantized_routed_expert_grouped_gb300 as m
    wl = synth.WORKLOADS["verify"]
    L = H.make_layer(wl, (synth.CB2, synth.NL4), 4, pool_experts=wl.E)
    B = H.make_bufs(L)
    call = H.expert_call(m, L, B)
    call.c.cap_entries = 4096  # 4096 * (2*768*4 + 24*36) bytes > the 4 MiB static buffer
    with pytest.raises(m.MoeError, match="-7"):
        call.call_static()
    assert np.isnan(B.out.cpu().numpy()).all()
