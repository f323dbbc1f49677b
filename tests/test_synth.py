"""The seeded generators: deterministic, device-independent by construction, right shapes and
distributions."""
import numpy as np
import torch

import synth


def test_mix64_matches_numpy_twin():
    k = synth.derive_key(3, 1, 4)
    idx = np.arange(0, 1 << 20, 997, dtype=np.int64)
    a = synth.mix64(k, torch.from_numpy(idx)).numpy().view(np.uint64)
    assert np.array_equal(a, synth.mix64_np(k, idx))


def test_weight_blobs_deterministic_and_sliceable():
    for typ in (synth.Q8_0, synth.Q4B, synth.NL4, synth.CB2, synth.CB3):
        w = synth.weight_blobs(typ, 16, 512, 3, 99)
        assert w.shape == (3, synth.blob_bytes(typ, 16, 512))
        w1 = synth.weight_blobs(typ, 16, 512, 1, 99, first_blob=2)
        assert torch.equal(w[2:], w1)
        assert not torch.equal(w[0], w[1])
        ub = {synth.Q8_0: 34, synth.Q4B: 20, synth.NL4: 18, synth.CB2: 70, synth.CB3: 102}[typ]
        u = w.numpy().reshape(-1, ub)
        d = u[:, 0:2].copy().view(np.float16).astype(np.float32)
        assert (d >= np.float16(1e-3)).all() and (d <= np.float16(1e-2)).all()
        if typ == synth.Q4B:
            m = u[:, 2:4].copy().view(np.float16).astype(np.float32)
            assert (m >= np.float16(-0.08)).all() and (m <= np.float16(-0.008)).all()
        if typ == synth.Q8_0:
            q = u[:, 2:].view(np.int8)
            assert q.min() >= -127 and q.max() <= 127


def test_small_inputs():
    g2, g3, t = synth.codebook(synth.CB2, 1), synth.codebook(synth.CB3, 1), synth.codebook(synth.NL4, 1)
    assert g2.shape == (256, 8) and set(np.unique(g2)) <= {-3, -1, 1, 3}
    assert g3.shape == (256, 4) and (g3 % 2 != 0).all() and np.abs(g3).max() <= 15
    assert t.shape == (16,) and (np.diff(t.astype(int)) > 0).all()
    r = synth.routing(4, 8, 64, 5)
    assert r.shape == (4, 8) and all(len(set(row)) == 8 for row in r)
    x = synth.activations(4, 2560, 5, outliers=0.01)
    assert x.dtype == np.float32 and x.shape == (4, 2560)
