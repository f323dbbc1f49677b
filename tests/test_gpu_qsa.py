"""QSA decode block scores (moe_qsa_block_scores) against the CPU oracle, bit for bit.

#2059 "QSA decode: the window's block scores with the queries in registers and six shuffles per
block" fixes the order of every fp32 step (the lane slices and their fused products, the warp
sum's pairings, relu, the head order, the tail's +1e9), so the GPU's scores must equal the
oracle's exactly: at small sizes on every block, at the page's 131k context on every block, and
at a 1M context on sampled blocks (a non-tail block's score depends on its own key and scale
only) plus the tail.
"""
import numpy as np
import pytest
import torch

import oracle_pins as P
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import quantized_routed_expert_grouped_gb300 as mod
    mod.lib()
    return mod


def _gpu(m, q, keys, scale):
    dev = "cuda"
    out = m.qsa_block_scores(torch.from_numpy(q).to(dev), torch.as_tensor(keys).to(dev),
                             torch.as_tensor(scale).to(dev))
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("n_blocks", [1, 2, 15, 16, 17, 63, 1000, 4097])
def test_qsa_scores_bitexact(m, orc, T, n_blocks):
    """Every block, ragged chunk tails (chunks hold 16 / 8 / 4 blocks at T = 1 / 2 / 3-4)."""
    q = synth.qsa_queries(T, 100 + T)
    keys, scale = synth.qsa_keys(n_blocks, 7 + n_blocks)
    got = _gpu(m, q, keys, scale)
    ref = orc.qsa_block_scores(q, keys.numpy(), scale.numpy())
    assert np.array_equal(_bits(got), _bits(ref))


def test_qsa_hand_worked_blocks(m, orc):
    """The oracle's hand-worked blocks (each value derived by hand from the page's order of
    operations) through the GPU."""
    q = np.zeros((1, 4, 128), np.float32)
    keys = np.zeros((6, 128), np.int8)
    scale = np.ones(6, np.float32)
    q[0, 0, 0], q[0, 0, 1] = -1.0, 1.0 + 2.0 ** -23
    keys[0, 0] = keys[0, 1] = 3
    q[0, 0, 4], q[0, 0, 5], q[0, 0, 6] = 2.0 ** -24, 2.0 ** -24, 1.0
    keys[1, 4] = keys[1, 5] = keys[1, 6] = 1
    q[0, 0, 8], q[0, 0, 12], q[0, 0, 76] = 2.0 ** 24, 1.0, 1.0
    keys[2, 8] = keys[2, 12] = keys[2, 76] = 1
    q[0, :, 16] = [1.0, 2.0 ** -24, 2.0 ** -24, 0.0]
    keys[3, 16] = 1
    q[0, 0, 20], q[0, 1, 20] = -3.0, 0.75
    keys[4, 20] = 2
    scale[4] = 4.0
    got = _gpu(m, q, keys, scale)[0]
    want = np.array([3 * 2.0 ** -23, 1 + 2.0 ** -23, 16777218.0, 1.0, 6.0, 1e9], np.float32)
    assert np.array_equal(_bits(got), _bits(want))
    P.check_qsa_hand(orc)  # the same values from the oracle


@pytest.mark.parametrize("T", [1, 4])
def test_qsa_131k_context(m, orc, T):
    """The page's context length (131k tokens: 32,768 full blocks of 4 tokens and the tail
    block), every block."""
    nb = synth.QSA_CONTEXTS["131k"]
    q = synth.qsa_queries(T, 31 + T)
    keys, scale = synth.qsa_keys(nb, 131)
    got = _gpu(m, q, keys, scale)
    ref = orc.qsa_block_scores(q, keys.numpy(), scale.numpy())
    assert np.array_equal(_bits(got), _bits(ref))
    assert (got[:, -1] >= 1e9).all() and (got[:, :-1] < 1e9).all()


@pytest.mark.parametrize("T", [2, 3, 4])
def test_qsa_1m_context_sampled(m, orc, T):
    """1M tokens (262,145 blocks), the launch the benchmark times: keys drawn on the device,
    4,096 sampled blocks and the tail recomputed by the oracle."""
    nb = synth.QSA_CONTEXTS["1M"]
    q = synth.qsa_queries(T, 77 + T)
    keys, scale = synth.qsa_keys(nb, 1000, device="cuda")
    got = m.qsa_block_scores(torch.from_numpy(q).cuda(), keys, scale)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    rng = np.random.Generator(np.random.PCG64(T))
    sample = np.sort(rng.choice(nb - 1, 4096, replace=False))
    kh, sh = keys.cpu().numpy(), scale.cpu().numpy()
    # the sampled non-tail blocks followed by a zero-key dummy tail (its score is not compared)
    ks = np.concatenate([kh[sample], np.zeros((1, 128), np.int8)])
    ss = np.concatenate([sh[sample], np.ones(1, np.float32)])
    ref = orc.qsa_block_scores(q, ks, ss)[:, :-1]
    assert np.array_equal(_bits(got[:, sample]), _bits(ref))
    # the tail: the oracle on the last block alone (a one-block pool is its own tail)
    ref_tail = orc.qsa_block_scores(q, kh[-1:], sh[-1:])[:, 0]
    assert np.array_equal(_bits(got[:, -1]), _bits(ref_tail))


def test_qsa_extreme_values(m, orc):
    """Keys at -128 and 127 (the whole int8 range converts exactly), large and tiny queries,
    negative dots (relu), subnormal products."""
    rng = np.random.Generator(np.random.PCG64(5))
    T, nb = 4, 40
    q = (rng.standard_normal((T, 4, 128)) * np.exp(rng.uniform(-80, 30, (T, 4, 128)))).astype(np.float32)
    keys = rng.choice(np.array([-128, -127, -1, 0, 1, 126, 127], np.int8), (nb, 128))
    scale = np.exp(rng.uniform(-20, 5, nb)).astype(np.float32)
    got = _gpu(m, q, keys, scale)
    ref = orc.qsa_block_scores(q, keys, scale)
    assert np.array_equal(_bits(got), _bits(ref))
