"""Shared helpers for the parity tests and the smoke check: build one seeded call (a layer of a
workload at window size T), run it through the C ABI, and run the CPU oracle on the same inputs.

The oracle's inputs come from the seeded generators (synth) or from the oracle itself, never
from the CUDA path.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch

import synth


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max|got - ref| / max|ref| (rows = leading axis)."""
    got = np.atleast_2d(got).astype(np.float64)
    ref = np.atleast_2d(ref).astype(np.float64)
    err = np.abs(got - ref).max(axis=1)
    scale = np.maximum(np.abs(ref).max(axis=1), 1e-30)
    return float((err / scale).max()) if len(err) else 0.0


@dataclass
class Layer:
    wl: synth.Workload
    gu_t: int
    dn_t: int
    T: int
    layer: int
    key_gu: int
    key_dn: int
    pool_gu: torch.Tensor      # [E, gu blob bytes] (device)
    pool_dn: torch.Tensor      # [E, down blob bytes] (device)
    tab_gu: torch.Tensor       # [E] int64 device pointers
    tab_dn: torch.Tensor
    cb_gu: np.ndarray | None
    cb_dn: np.ndarray | None
    cb_gu_d: torch.Tensor | None
    cb_dn_d: torch.Tensor | None
    x: np.ndarray              # fp32 [T, N]
    ids: np.ndarray            # int32 [T, k]


def pointer_table(pool: torch.Tensor) -> torch.Tensor:
    base, stride = pool.data_ptr(), pool.stride(0)
    return torch.tensor([base + i * stride for i in range(pool.shape[0])], dtype=torch.int64, device=pool.device)


def make_layer(wl: synth.Workload, pair, T: int, layer: int = 0, device="cuda", pool_experts=None) -> Layer:
    gu_t, dn_t = pair
    E, N, F = wl.E, wl.N, wl.F
    key_gu = synth.derive_key(wl.seed, layer, gu_t, 0)
    key_dn = synth.derive_key(wl.seed, layer, dn_t, 1)
    nE = E if pool_experts is None else pool_experts
    pool_gu = synth.weight_blobs(gu_t, 2 * F, N, nE, key_gu, device)
    pool_dn = synth.weight_blobs(dn_t, N, F, nE, key_dn, device)
    cb_gu = synth.codebook(gu_t, wl.seed * 7 + 1)
    cb_dn = synth.codebook(dn_t, wl.seed * 7 + 2)
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a).ravel()).to(device)
    x = synth.activations(T, N, wl.seed * 1000 + layer * 10 + T, wl.outliers)
    ids = synth.routing(T, wl.k, E, wl.seed * 1000 + layer * 10 + T + 5)
    return Layer(wl, gu_t, dn_t, T, layer, key_gu, key_dn, pool_gu, pool_dn, pointer_table(pool_gu),
                 pointer_table(pool_dn), cb_gu, cb_dn, dev(cb_gu), dev(cb_dn), x, ids)


def transcoded(m, L: Layer, dst_type: int, device="cuda") -> Layer:
    """A copy of layer L whose gate/up pool is the GPU's load-time transcoding of L's CB2/CB3 pool
    into the slot layout dst_type (the oracle keeps using L's native blobs: same integers)."""
    wl = L.wl
    rows = 2 * wl.F
    out = torch.zeros((L.pool_gu.shape[0], rows * synth.row_bytes(dst_type, wl.N)), dtype=torch.uint8, device=device)
    tab = pointer_table(out)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    m.transcode_cb(L.gu_t, L.cb_gu_d, dst_type, wl.N, rows, L.tab_gu, tab, err)
    assert int(err.item()) == 0
    return replace(L, gu_t=dst_type, pool_gu=out, tab_gu=tab, cb_gu_d=None)


def host_blobs(L: Layer, experts, role: str):
    """Host copies (regenerated on the CPU) of the given experts' blobs; dummies elsewhere."""
    wl = L.wl
    out = [np.zeros(1, np.uint8)] * wl.E
    for x in sorted(set(int(v) for v in experts)):
        if role == "gu":
            b = synth.weight_blobs(L.gu_t, 2 * wl.F, wl.N, 1, L.key_gu, "cpu", first_blob=x)
        else:
            b = synth.weight_blobs(L.dn_t, wl.N, wl.F, 1, L.key_dn, "cpu", first_blob=x)
        out[x] = b[0].numpy()
    return out


@dataclass
class Bufs:
    grp_expert: torch.Tensor
    grp_start: torch.Tensor
    n_groups: torch.Tensor
    ent_src: torch.Tensor
    ent_dst: torch.Tensor
    xq: torch.Tensor
    gu: torch.Tensor
    hq: torch.Tensor
    out: torch.Tensor
    err: torch.Tensor
    cap_groups: int
    cap_entries: int


def make_bufs(L: Layer, cap_entries=None, out_rows=None, device="cuda", fill=float("nan")) -> Bufs:
    wl = L.wl
    n = L.T * wl.k
    cap_e = cap_entries or n
    i32 = dict(dtype=torch.int32, device=device)
    return Bufs(
        grp_expert=torch.full((n,), -7, **i32), grp_start=torch.full((n + 1,), -7, **i32),
        n_groups=torch.zeros(1, **i32), ent_src=torch.full((cap_e,), -7, **i32),
        ent_dst=torch.full((cap_e,), -7, **i32),
        xq=torch.empty((L.T, wl.N // 32, 36), dtype=torch.uint8, device=device),
        gu=torch.full((cap_e, 2 * wl.F), fill, dtype=torch.float32, device=device),
        hq=torch.full((cap_e, wl.F // 32, 36), 0xA5, dtype=torch.uint8, device=device),
        out=torch.full((out_rows or n, wl.N), fill, dtype=torch.float32, device=device),
        err=torch.zeros(1, **i32), cap_groups=n, cap_entries=cap_e)


def gpu_route_and_quantize(m, L: Layer, B: Bufs, entry_base=0):
    ids = torch.from_numpy(L.ids).to(B.grp_expert.device)
    x = torch.from_numpy(L.x).to(B.grp_expert.device)
    m.route_group(ids, L.wl.E, entry_base, B.grp_expert, B.grp_start, B.n_groups, B.ent_src, B.ent_dst, B.err)
    m.quantize_q8_1(x, B.xq)


def expert_call(m, L: Layer, B: Bufs, grid_groups=0, flags=1):
    wl = L.wl
    return m.ExpertCall(L.gu_t, L.cb_gu_d, L.dn_t, L.cb_dn_d, wl.N, wl.F, L.tab_gu, L.tab_dn, wl.E,
                        B.grp_expert, B.grp_start, B.n_groups, B.cap_groups, grid_groups, B.cap_entries, B.xq,
                        B.ent_src, B.ent_dst, B.gu, B.hq, B.out, B.err, flags)


def oracle_call(o, L: Layer, r=None, gu_blobs=None, dn_blobs=None):
    """The whole call on the CPU from x: routing, q8_1, gate/up (fp64), SwiGLU + q8_1 on the
    fp32-rounded gate/up, down (fp64). Returns a dict of every stage."""
    wl = L.wl
    n = L.T * wl.k
    r = r or o.route_group(L.ids, wl.E)
    G = r["n_groups"]
    gu_blobs = gu_blobs or host_blobs(L, r["grp_expert"], "gu")
    dn_blobs = dn_blobs or host_blobs(L, r["grp_expert"], "dn")
    xq = o.quantize_q8_1(L.x)
    gu = np.full((n, 2 * wl.F), np.nan)
    o.grouped_gemv(L.gu_t, wl.N, 2 * wl.F, gu_blobs, r["grp_expert"], r["grp_start"], G, xq,
                   ent_in=r["ent_src"], out=gu, cb=L.cb_gu)
    hq = np.zeros((n, wl.F // 32, 36), np.uint8)
    o.swiglu_q8_1(gu.astype(np.float32), wl.F, r["grp_start"][0], r["grp_start"][G], hq)
    out = np.full((n, wl.N), np.nan)
    o.grouped_gemv(L.dn_t, wl.F, wl.N, dn_blobs, r["grp_expert"], r["grp_start"], G, hq,
                   ent_out=r["ent_dst"], out=out, cb=L.cb_dn)
    return dict(route=r, xq=xq, gu=gu, hq=hq, out=out, gu_blobs=gu_blobs, dn_blobs=dn_blobs)


def q8_1_code_flips(a: np.ndarray, b: np.ndarray):
    """(number of differing codes, number of differing d/s fields) between two q8_1 arrays."""
    a = a.reshape(-1, 36)
    b = b.reshape(-1, 36)
    return int((a[:, 4:] != b[:, 4:]).sum()), int((a[:, :4] != b[:, :4]).any(axis=1).sum())
