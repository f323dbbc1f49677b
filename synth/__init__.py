"""Seeded synthetic inputs for the grouped routed-expert decode.

This module holds no arithmetic of the method: it only draws random bytes, scales,
codebooks, activations and routings with the distributions of the workloads, and knows where
the scale fields sit inside each format's blocks. Both the CUDA path's tests/benchmark and
the CPU oracle take their inputs from here.

Weight blobs come from a counter-based generator (the SplitMix64 output function of Steele,
Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014, applied to
key + (i+1) * golden gamma) written with torch integer ops, so the same bytes come out on the
CPU and on the GPU: large pools are drawn on the device, and any one expert can be redrawn on
the host for the oracle. Activations, codebooks and routings are small and drawn with numpy.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

Q8_0, Q4B, NL4, CB2, CB3, CB3X, CB2X = 1, 2, 3, 4, 5, 6, 7
NAMES = {Q8_0: "Q8_0", Q4B: "Q4B", NL4: "NL4", CB2: "CB2", CB3: "CB3", CB3X: "CB3X", CB2X: "CB2X"}
BY_NAME = {v: k for k, v in NAMES.items()}

# (bytes per unit, weights per unit, [(field offset, distribution)]) per format
_UNIT = {
    Q8_0: (34, 32, [(0, "d")]),
    Q4B: (20, 32, [(0, "d"), (2, "m")]),
    NL4: (18, 32, [(0, "d")]),
    CB2: (70, 256, [(0, "d")]),
    CB3: (102, 256, [(0, "d")]),
}
_DIST = {"d": (1e-3, 1e-2), "m": (-0.08, -0.008)}


# bytes per 256 weights of the transcoded slot layouts (codes + 8-byte scale record)
_SLOT = {CB3X: 136, CB2X: 72}


def row_bytes(typ: int, K: int) -> int:
    if typ in _SLOT:
        assert K % 256 == 0
        return K // 256 * _SLOT[typ]
    ub, uw, _ = _UNIT[typ]
    assert K % uw == 0
    return K // uw * ub


def blob_bytes(typ: int, rows: int, K: int) -> int:
    return rows * row_bytes(typ, K)


# ---------------------------------------------------------------- counter-based generator

_M64 = (1 << 64) - 1


def _s64(c: int) -> int:
    c &= _M64
    return c - (1 << 64) if c >> 63 else c


_GAMMA = _s64(0x9E3779B97F4A7C15)
_MUL1 = _s64(0xBF58476D1CE4E5B9)
_MUL2 = _s64(0x94D049BB133111EB)


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    return (z >> s) & ((1 << (64 - s)) - 1)


def mix64(key, idx: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output for counters idx (int64 tensor) under a 64-bit key (an int, or an
    int64 tensor that broadcasts against idx)."""
    z = idx.to(torch.int64) + 1
    z = z * _GAMMA + (_s64(key) if isinstance(key, int) else key)
    z = (z ^ _srl(z, 30)) * _MUL1
    z = (z ^ _srl(z, 27)) * _MUL2
    return z ^ _srl(z, 31)


def mix64_np(key: int, idx: np.ndarray) -> np.ndarray:
    """numpy twin of mix64 (uint64 wrap-around arithmetic), for cross-checks."""
    with np.errstate(over="ignore"):
        z = idx.astype(np.uint64) + np.uint64(1)
        z = z * np.uint64(0x9E3779B97F4A7C15) + np.uint64(key & _M64)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def derive_key(*parts: int) -> int:
    """64-bit key from a tuple of small integers (seed, layer, expert, role ...)."""
    k = 0x243F6A8885A308D3
    for p in parts:
        k = int(mix64(k, torch.tensor([p & 0xFFFFFFFF], dtype=torch.int64))[0]) & _M64
    return k


def _blob_key(key: int, blob: int, part: int) -> int:
    return derive_key(key & 0xFFFFFFFF, key >> 32, blob, part)


def weight_blobs(typ: int, rows: int, K: int, n_blobs: int, key: int, device="cpu",
                 first_blob: int = 0, chunk_bytes: int = 1 << 28) -> torch.Tensor:
    """uint8 [n_blobs, rows*row_bytes]: blob b is expert first_blob+b of the pool `key`.

    Index bytes, sign bytes, sub-scale nibbles and 4-bit codes are uniform random bytes;
    Q8_0 weights are (byte % 255) - 127 (uniform in [-127, 127] up to a 1/256 bias at -127);
    scales d / D are fp16 uniform in [1e-3, 1e-2], Q4B minimums m fp16 uniform in
    [-0.08, -0.008]. A 24-bit uniform u becomes lo + u*(hi-lo) in fp32, then fp16."""
    ub, uw, fields = _UNIT[typ]
    nbytes = blob_bytes(typ, rows, K)
    nunits = nbytes // ub
    nwords = (nbytes + 7) // 8
    out = torch.empty((n_blobs, nbytes), dtype=torch.uint8, device=device)
    step = max(1, chunk_bytes // (nwords * 8 * 4))
    iw = torch.arange(nwords, device=device, dtype=torch.int64)
    iu = torch.arange(nunits, device=device, dtype=torch.int64)
    for b0 in range(0, n_blobs, step):
        nb = min(step, n_blobs - b0)
        blobs = range(first_blob + b0, first_blob + b0 + nb)
        kb = torch.tensor([_s64(_blob_key(key, b, 0)) for b in blobs], dtype=torch.int64, device=device)
        by = mix64(kb[:, None], iw[None, :]).view(torch.uint8).view(nb, nwords * 8)[:, :nbytes]
        if typ == Q8_0:
            by = ((by.to(torch.int16) % 255) - 127).to(torch.int8).view(torch.uint8)
        units = by.reshape(nb, nunits, ub).clone()
        for fi, (off, dist) in enumerate(fields):
            lo, hi = _DIST[dist]
            ks = torch.tensor([_s64(_blob_key(key, b, 1 + fi)) for b in blobs], dtype=torch.int64,
                              device=device)
            h = mix64(ks[:, None], iu[None, :])
            u = _srl(h, 40).to(torch.float32) * float(2.0 ** -24)
            v = u * torch.tensor(hi - lo, dtype=torch.float32, device=device)
            v = v + torch.tensor(lo, dtype=torch.float32, device=device)
            units[:, :, off:off + 2] = v.to(torch.float16).view(torch.uint8).view(nb, nunits, 2)
        out[b0:b0 + nb] = units.view(nb, nbytes)
    return out


# ---------------------------------------------------------------- small host-side inputs

def codebook(typ: int, seed: int):
    """CB2: 256x8 int8 in {-3,-1,1,3}; CB3: 256x4 int8 odd in [-15,15]; NL4: 16 distinct
    sorted int8 in [-127,127]; None for the formats without one."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if typ == CB2:
        return rng.choice(np.array([-3, -1, 1, 3], dtype=np.int8), size=(256, 8))
    if typ == CB3:
        return rng.choice(np.arange(-15, 16, 2, dtype=np.int8), size=(256, 4))
    if typ == NL4:
        return np.sort(rng.choice(np.arange(-127, 128, dtype=np.int16), 16, replace=False)).astype(np.int8)
    return None


def activations(T: int, N: int, seed: int, outliers: float = 0.0) -> np.ndarray:
    """fp32 [T, N] N(0,1); a fraction `outliers` of the elements multiplied by 20."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((T, N)).astype(np.float32)
    if outliers > 0:
        m = rng.random((T, N)) < outliers
        x[m] *= np.float32(20.0)
    return x


def routing(T: int, k: int, E: int, seed: int) -> np.ndarray:
    """int32 [T, k]: k distinct expert ids per token, uniform."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


# ---------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    T: tuple
    E: int
    k: int
    N: int
    F: int
    pairs: tuple            # ((gate/up type, down type), ...)
    outliers: float = 0.0
    seed: int = 1
    second_call: bool = False
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", 1, (1,), 8, 2, 512, 256, ((Q8_0, Q8_0),), seed=11),
    "verify": Workload("verify", 1, (4,), 64, 8, 2560, 768, ((CB2, NL4),), seed=22),
    "window48": Workload("window48", 48, (1, 2, 3, 4), 128, 8, 2560, 768, ((CB3, NL4),), seed=33),
    "sparse": Workload("sparse", 1, (4,), 64, 8, 2560, 768, ((CB2, NL4),), seed=44, second_call=True),
    "sweep": Workload("sweep", 1, (4,), 256, 8, 4096, 1536,
                      tuple((g, d) for g in (Q8_0, Q4B, CB2, CB3) for d in (NL4, Q8_0)),
                      outliers=0.01, seed=55),
}


# ---------------------------------------------------------------- QSA decode block scores
QSA_HEADS, QSA_DIM = 4, 128
# contexts of the page's measurements and a longer one: 131k tokens in blocks of 4 tokens plus
# the tail block (32,769 blocks), and 1M tokens
QSA_CONTEXTS = {"131k": 32769, "1M": 262145}


def qsa_queries(T: int, seed: int) -> np.ndarray:
    """The window's T queries, fp32 [T, 4 heads, 128], N(0, 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal((T, QSA_HEADS, QSA_DIM)).astype(np.float32)


def qsa_keys(n_blocks: int, seed: int, device="cpu", first_block: int = 0):
    """Pooled int8 keys [n_blocks, 128], uniform in [-127, 127], and fp32 scales [n_blocks],
    uniform in [1e-3, 1e-2], from the counter-based generator (the same values on any device;
    first_block selects a window of a larger pool)."""
    idx = torch.arange(first_block * QSA_DIM, (first_block + n_blocks) * QSA_DIM, dtype=torch.int64, device=device)
    z = mix64(seed, idx)
    keys = ((_srl(z, 32) % 255) - 127).to(torch.int8).view(n_blocks, QSA_DIM)
    bi = torch.arange(first_block, first_block + n_blocks, dtype=torch.int64, device=device)
    u = _srl(mix64(seed ^ 0x5CA1E, bi), 40).to(torch.float64) / float(1 << 24)
    scale = (1e-3 + u * (1e-2 - 1e-3)).to(torch.float32)
    return keys, scale
