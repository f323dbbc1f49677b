"""The steps either side of the grouped call on the GPU against the CPU oracle: the router's top-k
ids (bit for bit, ties included) and softmax weights (max|err| / max|ref| <= 1e-5 per token), the
per-token weighted combine (same bar), and one whole MoE block: logits -> router -> grouped
expert call -> combine, against the oracle's chain."""
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


def _logits(T, E, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0, E // 2] = lg[0, E // 3]          # a tie between two experts
    if T > 1:
        lg[1, :] = np.float32(0.125)       # every expert tied
    if T > 2:
        lg[2, ::3] = np.float32(4.0)       # many tied at the top
    return lg


@pytest.mark.parametrize("T,E,k", [(4, 8, 2), (4, 64, 8), (4, 128, 8), (4, 256, 8), (7, 1000, 32), (3, 32, 32)])
def test_router_topk_matches_oracle(m, orc, T, E, k):
    lg = _logits(T, E, 1000 * E + k)
    ids, w = m.router_topk(torch.from_numpy(lg).cuda(), k)
    torch.cuda.synchronize()
    ref_ids, ref_w, rc = orc.router_topk(lg, k)
    assert rc == 0
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    got = w.cpu().numpy().astype(np.float64)
    for t in range(T):
        assert np.abs(got[t] - ref_w[t]).max() / np.abs(ref_w[t]).max() <= TOL


def test_combine_matches_oracle_and_skips_dropped(m, orc):
    rng = np.random.Generator(np.random.PCG64(77))
    T, k, E, N = 4, 8, 128, 2560
    out = rng.standard_normal((T * k, N)).astype(np.float32)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[0, 3] = -1
    ids[2, 7] = E + 5
    for t, j in ((0, 3), (2, 7)):
        out[t * k + j] = np.nan  # a dropped entry's row is never written: it must not be read
    w = rng.random((T, k)).astype(np.float32)
    y = m.combine(torch.from_numpy(out).cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), E)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    ref = orc.combine(out, ids, w.astype(np.float64), E)
    assert np.isfinite(got).all()
    assert H.rel_err(got, ref) <= TOL


def test_moe_block_end_to_end(m, orc):
    """Router logits -> top-k and weights (GPU) -> grouped expert call on the window's layer 0
    geometry at T = 4 (CB3 gate/up, NL4 down) -> combine (GPU), against the oracle's router,
    grouped call (from x, fp64) and combine."""
    wl = synth.WORKLOADS["window48"]
    L0 = H.make_layer(wl, (synth.CB3, synth.NL4), 4)
    lg = _logits(4, wl.E, 4242)
    ids, w = m.router_topk(torch.from_numpy(lg).cuda(), wl.k)
    torch.cuda.synchronize()
    ref_ids, ref_w, rc = orc.router_topk(lg, wl.k)
    assert rc == 0 and np.array_equal(ids.cpu().numpy(), ref_ids)
    L = H.Layer(**{**L0.__dict__, "ids": ref_ids})
    B = H.make_bufs(L)
    H.gpu_route_and_quantize(m, L, B)
    H.expert_call(m, L, B)()
    y = m.combine(B.out, ids, w, wl.E)
    torch.cuda.synchronize()
    assert int(B.err.item()) == 0
    ref = H.oracle_call(orc, L)
    flips, scale_diffs = H.q8_1_code_flips(B.hq.cpu().numpy(), ref["hq"])
    y_ref = orc.combine(ref["out"].astype(np.float32), ref_ids, ref_w, wl.E)
    err = H.rel_err(y.cpu().numpy(), y_ref)
    assert err <= (TOL if flips == 0 and scale_diffs == 0 else 2e-3), (err, flips)
