"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each check_* takes an ``oracle.Oracle`` and raises AssertionError on a mismatch. They are run
on the real oracle (tests/test_oracle_pins.py) and on builds with planted mistakes
(tests/test_oracle_mutants.py), which each must fail at least one check.

What pins what:
  binary16      -> numpy's IEEE binary16 conversion (a library routine), all 65536 patterns,
                   every rounding midpoint and random values
  exp/silu      -> fp64 exp from numpy (<= 2 ulp), special values
  q8_1          -> closed forms (zero and constant blocks, halfway cases rounded away from
                   zero), s16 == binary16(fp32(d) * sum q) with numpy's own arithmetic,
                   the rounding bound |x - d q| <= d/2
  formats       -> hand-built blocks with hand-worked weights (every field, nibble order, sign
                   bit order, sub-scale nibble and 2*sub+1), one-hot activations that read out
                   one column, and brute-force fp64 dot products of dequantized operands
  grouping      -> a hand-worked routing example and invariants on random routings
  router        -> a hand-worked top-k with a tie and its softmax in closed form (e/(e+2),
                   1/(e+2)), equal logits (ids 0..k-1, weights 1/k), and on random logits: no
                   unselected logit ranks above a selected one, weights sum to 1, weight ratios
                   are e^(l_i - l_j)
  combine       -> one-hot weights read out one row, identical rows give the row times the weight
                   sum, a hand-worked 2-token example, dropped ids skipped
  grouped steps -> permutation invariants and untouched rows
  QSA scores    -> hand-worked blocks whose exact fp32 values pin each step's order (the fused
                   in-lane products, 4 consecutive dims per lane, the warp-sum pairings, the head
                   order, relu after the scale, +1e9 on the tail only), and fp64 brute force within
                   a stated rounding bound; queries and non-tail blocks independent
"""
from __future__ import annotations

import numpy as np

Q8_0, Q4B, NL4, CB2, CB3, CB3X, CB2X = 1, 2, 3, 4, 5, 6, 7


def _h(v):
    return int(np.array(v, dtype=np.float16).view(np.uint16))


def _wr16(buf, off, bits):
    buf[off] = bits & 255
    buf[off + 1] = bits >> 8


# ------------------------------------------------------------------ binary16

def check_f16(o):
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = o.h2f(allh)
    ref = allh.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(f), nan)
    assert np.array_equal(f[~nan].view(np.uint32), ref[~nan].view(np.uint32)), "h2f"
    # every finite binary16 value, every midpoint between neighbours (ties), and random floats
    fin = ref[np.isfinite(ref) & (ref >= 0)].astype(np.float64)
    fin = np.unique(fin)
    mids = ((fin[:-1] + fin[1:]) / 2).astype(np.float32)
    rng = np.random.Generator(np.random.PCG64(7))
    rnd = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 12, 20000))).astype(np.float32)
    xs = np.concatenate([fin.astype(np.float32), mids, -mids, rnd,
                         np.array([65504, 65519.99, 65520, 1e30, -1e30, 0.0, -0.0, 2.0 ** -25,
                                   3 * 2.0 ** -26, 2.0 ** -26], np.float32)])
    got = o.f2h(xs)
    with np.errstate(over="ignore"):
        exp = xs.astype(np.float16).view(np.uint16)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, f"f2h mismatch at {xs[bad[:5]]}: {got[bad[:5]]} vs {exp[bad[:5]]}"


# ------------------------------------------------------------------ exp, silu, swiglu

def _ulps(got, ref64):
    ref32 = ref64.astype(np.float32)
    sp = np.spacing(np.abs(ref32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - ref64) / sp


def check_exp(o):
    x = np.concatenate([np.linspace(-103.0, 88.7, 40001), np.linspace(-1, 1, 4001),
                        np.array([0.0, 1e-10, -1e-10, 0.34657359, -0.34657359])]).astype(np.float32)
    e = o.expf(x)
    ref = np.exp(x.astype(np.float64))
    m = ref > 2.0 ** -126  # normal results: ulp bound; subnormal results: absolute bound
    assert np.max(_ulps(e[m], ref[m])) <= 2.0, "exp ulp error"
    assert np.max(np.abs(e[~m] - ref[~m])) <= 2.0 ** -149
    sp = o.expf(np.array([0.0, 89.0, 100.0, -105.0, -1000.0, np.nan], np.float32))
    assert sp[0] == 1.0 and np.isinf(sp[1]) and np.isinf(sp[2]) and sp[3] == 0 and sp[4] == 0
    assert np.isnan(sp[5])


def check_silu(o):
    g = np.concatenate([np.linspace(-30, 30, 6001), np.linspace(-1e-3, 1e-3, 101)]).astype(np.float32)
    s = o.silu(g)
    g64 = g.astype(np.float64)
    ref = g64 / (1.0 + np.exp(-g64))
    nz = np.abs(ref) > 1e-30
    assert np.max(_ulps(s[nz], ref[nz])) <= 4.0, "silu"
    sp = o.silu(np.array([0.0, -200.0, 200.0, -89.0], np.float32))
    assert sp[0] == 0.0 and not np.signbit(sp[0])
    assert sp[1] == 0.0 and np.signbit(sp[1]), "silu(-large) is -0"
    assert sp[2] == 200.0
    # the product is one fp32 rounding of silu(g) * u (#363, "What changes")
    rng = np.random.Generator(np.random.PCG64(3))
    gg = rng.standard_normal(2000).astype(np.float32) * 4
    uu = rng.standard_normal(2000).astype(np.float32) * 4
    h = o.swiglu(gg, uu)
    ref = gg.astype(np.float64) / (1 + np.exp(-gg.astype(np.float64))) * uu.astype(np.float64)
    nz = np.abs(ref) > 1e-30
    assert np.max(_ulps(h[nz], ref[nz])) <= 5.0, "swiglu"


# ------------------------------------------------------------------ q8_1

def _parse_q8_1(blocks):
    b = blocks.reshape(-1, 36)
    d = b[:, 0:2].copy().view(np.float16).astype(np.float64).ravel()
    s = b[:, 2:4].copy().view(np.float16).astype(np.float64).ravel()
    q = b[:, 4:].view(np.int8).astype(np.int64)
    return d, s, q, b[:, 0:2].copy().view(np.uint16).ravel(), b[:, 2:4].copy().view(np.uint16).ravel()


def check_q8_1(o):
    # zero block, constant blocks, and a block with halfway cases (d = 1 exactly)
    half = np.zeros(32, np.float32)
    half[:8] = [127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5]
    x = np.stack([np.zeros(32, np.float32), np.full(32, 3.0, np.float32), np.full(32, -0.02, np.float32), half])
    d, s, q, d16, s16 = _parse_q8_1(o.quantize_q8_1(x))
    assert d16[0] == 0 and s16[0] == 0 and not q[0].any()
    assert (q[1] == 127).all() and d16[1] == _h(np.float32(3.0) / np.float32(127))
    assert (q[2] == -127).all() and d16[2] == _h(np.float32(0.02) / np.float32(127))
    assert list(q[3][:8]) == [127, 3, -3, 1, -1, 2, -2, 127] and d16[3] == _h(1.0), "round half away"
    assert s16[3] == _h(np.float32(sum(q[3])))
    # random rows: the definition of s, the rounding bound, the code range
    rng = np.random.Generator(np.random.PCG64(5))
    x = rng.standard_normal((64, 256)).astype(np.float32) * np.exp(rng.uniform(-6, 6, (64, 1))).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 20
    d, s, q, d16, s16 = _parse_q8_1(o.quantize_q8_1(x))
    xb = x.reshape(-1, 32)
    amax = np.max(np.abs(xb), axis=1)
    d32 = amax / np.float32(127)
    assert np.array_equal(d16, d32.astype(np.float16).view(np.uint16)), "d16"
    S = q.sum(axis=1)
    assert np.array_equal(s16, (d32 * S.astype(np.float32)).astype(np.float32).astype(np.float16).view(np.uint16)), "s16"
    assert np.abs(q).max() <= 127 and (np.abs(q).max(axis=1) == 127).all()
    err = np.abs(xb.astype(np.float64) - d32.astype(np.float64)[:, None] * q)
    assert (err <= d32.astype(np.float64)[:, None] * 0.5 * (1 + 1e-6)).all(), "rounding bound"


# ------------------------------------------------------------------ formats: hand-built blocks

def check_formats_hand(o):
    # Q4B: d = 0.25, m = -1; qs[0] = 0x21 -> codes 1 (w0) and 2 (w16); qs[15] = 0xF0 -> 0 (w15), 15 (w31)
    blk = np.zeros(20, np.uint8)
    _wr16(blk, 0, _h(0.25)); _wr16(blk, 2, _h(-1.0))
    blk[4 + 0] = 0x21; blk[4 + 15] = 0xF0
    w = o.dequant_row(Q4B, blk, 32)
    exp = np.full(32, -1.0); exp[0] = -0.75; exp[16] = -0.5; exp[15] = -1.0; exp[31] = 2.75
    assert np.array_equal(w, exp), f"Q4B {w}"
    # NL4: d = 2, table = -120 + 15 j; qs[3] = 0x5A -> code 10 (w3), 5 (w19)
    tab = np.array([-120 + 15 * j for j in range(16)], np.int8)
    blk = np.zeros(18, np.uint8)
    _wr16(blk, 0, _h(2.0)); blk[2 + 3] = 0x5A
    w = o.dequant_row(NL4, blk, 32, tab)
    exp = np.full(32, 2.0 * -120); exp[3] = 2.0 * 30; exp[19] = 2.0 * -45
    assert np.array_equal(w, exp), f"NL4 {w}"
    # Q8_0: d = 0.5, q = -16..15
    blk = np.zeros(34, np.uint8)
    _wr16(blk, 0, _h(0.5)); blk[2:] = np.arange(-16, 16, dtype=np.int8).view(np.uint8)
    assert np.array_equal(o.dequant_row(Q8_0, blk, 32), 0.5 * np.arange(-16, 16)), "Q8_0"
    # CB2: D = 0.5; grid2[9] = [1,3,-1,-3,3,1,-3,-1], all other rows +1
    g2 = np.ones((256, 8), np.int8); g2[9] = [1, 3, -1, -3, 3, 1, -3, -1]
    sb = np.zeros(70, np.uint8)
    _wr16(sb, 0, _h(0.5))
    sb[2 + 0] = 9; sb[34 + 0] = 0b10000001           # group 0: bits 0 and 7 negate weights 0, 7
    sb[2 + 4] = 9                                    # group 4 = weights 32..39 (sub-block 1)
    sb[2 + 28] = 9; sb[34 + 28] = 0x10               # group 28 = weights 224..231, weight 228 negated
    sb[66 + 0] = 0x52                                # sub_0 = 2 (ls 5), sub_1 = 5 (ls 11)
    sb[66 + 3] = 0xE0                                # sub_6 = 0 (ls 1), sub_7 = 14 (ls 29)
    w = o.dequant_row(CB2, sb, 256, g2)
    assert list(w[0:8]) == [-2.5, 7.5, -2.5, -7.5, 7.5, 2.5, -7.5, 2.5], f"CB2 g0 {w[0:8]}"
    assert list(w[8:10]) == [2.5, 2.5]
    assert list(w[32:40]) == [5.5 * v for v in [1, 3, -1, -3, 3, 1, -3, -1]], f"CB2 g4 {w[32:40]}"
    assert list(w[224:232]) == [14.5 * v for v in [1, 3, -1, -3, -3, 1, -3, -1]], f"CB2 g28 {w[224:232]}"
    assert w[192] == 0.5 and w[100] == 0.5
    # CB3: D = 1; grid3[7] = [1,3,5,7], all other rows +1
    g3 = np.ones((256, 4), np.int8); g3[7] = [1, 3, 5, 7]
    sb = np.zeros(102, np.uint8)
    _wr16(sb, 0, _h(1.0))
    sb[2 + 0] = 7; sb[2 + 1] = 7; sb[66 + 0] = 0x42  # weights 0..7: bits 1 and 6 negate weights 1, 6
    sb[2 + 40] = 7; sb[66 + 20] = 0x08               # group 40 = weights 160..163; weight 163 negated
    sb[98 + 0] = 0x03                                # sub_0 = 3 (ls 7), sub_1 = 0 (ls 1)
    sb[98 + 2] = 0x90                                # sub_4 = 0, sub_5 = 9 (ls 19)
    w = o.dequant_row(CB3, sb, 256, g3)
    assert list(w[0:8]) == [7, -21, 35, 49, 7, 21, -35, 49], f"CB3 {w[0:8]}"
    assert list(w[160:164]) == [19, 57, 95, -133], f"CB3 g40 {w[160:164]}"
    assert w[32] == 1 and w[164] == 19 and w[255] == 1


def _random_row(typ, K, rng):
    per = {Q8_0: 34, Q4B: 20, NL4: 18}.get(typ)
    if per:
        row = rng.integers(0, 256, (K // 32) * per, dtype=np.uint8)
        units = row.reshape(-1, per)
        sc = rng.uniform(1e-3, 1e-2, len(units)).astype(np.float16).view(np.uint16)
        units[:, 0] = sc & 255; units[:, 1] = sc >> 8
        if typ == Q4B:
            mm = rng.uniform(-0.08, -0.008, len(units)).astype(np.float16).view(np.uint16)
            units[:, 2] = mm & 255; units[:, 3] = mm >> 8
        if typ == Q8_0:
            q = units[:, 2:].view(np.int8)
            q[q == -128] = -127
        return row
    per = 70 if typ == CB2 else 102
    row = rng.integers(0, 256, (K // 256) * per, dtype=np.uint8)
    units = row.reshape(-1, per)
    sc = rng.uniform(1e-3, 1e-2, len(units)).astype(np.float16).view(np.uint16)
    units[:, 0] = sc & 255; units[:, 1] = sc >> 8
    return row


def _cb_for(typ, rng):
    if typ == CB2:
        return rng.choice(np.array([-3, -1, 1, 3], np.int8), (256, 8))
    if typ == CB3:
        return rng.choice(np.arange(-15, 16, 2).astype(np.int8), (256, 4))
    if typ == NL4:
        return np.sort(rng.choice(np.arange(-127, 128), 16, replace=False)).astype(np.int8)
    return None


def check_formats_onehot(o):
    """x = c e_j gives a q8_1 row with one code 127: the block sum reads out column j."""
    rng = np.random.Generator(np.random.PCG64(9))
    K = 512
    for typ in (Q8_0, Q4B, NL4, CB2, CB3):
        cb = _cb_for(typ, rng)
        row = _random_row(typ, K, rng)
        w = o.dequant_row(typ, row, K, cb)
        for j in (0, 1, 7, 31, 32, 100, 255, 256, 300, 511):
            x = np.zeros((1, K), np.float32); x[0, j] = 1.27
            xq = o.quantize_q8_1(x)[0]
            d = float(np.float16(np.float32(1.27) / np.float32(127)))
            got = o.row_dot(typ, row, K, xq, cb)
            if typ == Q4B:  # every block adds m * s_x; only block j//32 has s_x != 0
                b = j // 32
                m = float(row[20 * b + 2:20 * b + 4].copy().view(np.float16)[0])
                dw = float(row[20 * b:20 * b + 2].copy().view(np.float16)[0])
                s = float(np.float16(np.float32(np.float32(1.27) / np.float32(127)) * np.float32(127)))
                want = dw * (w[j] - m) / dw * d * 127 + m * s
            else:
                want = w[j] * d * 127
            assert abs(got - want) <= 1e-12 * max(1.0, abs(want)), (typ, j, got, want)


def check_formats_bruteforce(o):
    """Blocked integer formula == fp64 dot of the dequantized weights and activations."""
    rng = np.random.Generator(np.random.PCG64(13))
    K = 512
    for typ in (Q8_0, Q4B, NL4, CB2, CB3):
        cb = _cb_for(typ, rng)
        for _ in range(6):
            row = _random_row(typ, K, rng)
            x = rng.standard_normal((1, K)).astype(np.float32)
            xq = o.quantize_q8_1(x)[0]
            d, s, q, _, _ = _parse_q8_1(xq)
            xd = (d[:, None] * q).ravel()
            w = o.dequant_row(typ, row, K, cb)
            brute = float(np.dot(w, xd))
            got = o.row_dot(typ, row, K, xq, cb)
            tol = 1e-12 * np.sum(np.abs(w * xd))
            if typ == Q4B:  # the m term uses the stored s16 instead of d16 * sum q
                m = row.reshape(-1, 20)[:, 2:4].copy().view(np.float16).astype(np.float64).ravel()
                tol += float(np.sum(np.abs(m) * np.abs(s - d * q.sum(axis=1))))
            assert abs(got - brute) <= tol, (typ, got, brute, tol)
            # per-block integer sums agree with a direct int64 sum over the integer weights
            v = o.int_weights(typ, row, K, cb).astype(np.int64)
            isum = o.block_isum(typ, row, K, xq, cb)
            assert np.array_equal(isum, (v.reshape(-1, 32) * q).sum(axis=1))


# ------------------------------------------------------------------ transcoded slot layouts

def check_slots(o):
    """Load-time slot layouts hold exactly the native integers and scales (round trip through
    the native decode), in the documented byte positions (hand-worked), and refuse values that
    do not fit."""
    rng = np.random.Generator(np.random.PCG64(29))
    K = 512
    for src, dst in ((CB3, CB3X), (CB2, CB2X), (CB2, CB3X)):
        cb = _cb_for(src, rng)
        for _ in range(4):
            row = _random_row(src, K, rng)
            t, rc = o.transcode_row(src, row, K, cb, dst)
            assert rc == 0 and len(t) == o.row_bytes(dst, K)
            assert np.array_equal(o.int_weights(dst, t, K), o.int_weights(src, row, K, cb)), (src, dst)
            assert np.array_equal(o.dequant_row(dst, t, K), o.dequant_row(src, row, K, cb))
            x = rng.standard_normal((1, K)).astype(np.float32)
            xq = o.quantize_q8_1(x)[0]
            assert np.array_equal(o.block_isum(dst, t, K, xq), o.block_isum(src, row, K, xq, cb))
            assert o.row_dot(dst, t, K, xq) == o.row_dot(src, row, K, xq, cb)
    # hand-worked CB3X bytes: CB3 weights 0..3 = +1 -3 +5 +7, weight 16 = -15, weight 17 = +15
    g3 = np.ones((256, 4), np.int8); g3[7] = [1, 3, 5, 7]; g3[9] = [15, 15, 1, 1]
    sb = np.zeros(102, np.uint8)
    _wr16(sb, 0, _h(0.5))
    sb[2 + 0] = 7; sb[66 + 0] = 0x02          # weight 1 negated
    sb[2 + 4] = 9; sb[66 + 2] = 0x01          # group 4 = weights 16..19, weight 16 negated
    sb[98:102] = [0x21, 0x43, 0x65, 0x87]
    t, rc = o.transcode_row(CB3, sb, 256, g3, CB3X)
    assert rc == 0
    # u = (v-1)/2 + 8: +1 -> 8, -3 -> 6, +5 -> 10, +7 -> 11, -15 -> 0, +15 -> 15, +1 -> 8
    assert list(t[0:4]) == [8 | (0 << 4), 6 | (15 << 4), 10 | (8 << 4), 11 | (8 << 4)], list(t[0:4])
    assert list(t[128:136]) == [sb[0], sb[1], 0, 0, 0x21, 0x43, 0x65, 0x87]
    # hand-worked CB2X bytes: CB2 group 0 = weights 0..7 from grid2[5] = [3,-3,1,-1,3,3,-1,1]
    g2 = np.ones((256, 8), np.int8); g2[5] = [3, -3, 1, -1, 3, 3, -1, 1]
    sb = np.zeros(70, np.uint8)
    sb[2 + 0] = 5; sb[34 + 0] = 0x80          # weight 7 negated -> -1
    t, rc = o.transcode_row(CB2, sb, 256, g2, CB2X)
    assert rc == 0
    # u = (v-1)/2 + 2: 3 -> 3, -3 -> 0, 1 -> 2, -1 -> 1; weights 0..7 sit in bits 0-1 of bytes 0..7
    assert [int(v) & 3 for v in t[0:8]] == [3, 0, 2, 1, 3, 3, 1, 1], [int(v) & 3 for v in t[0:8]]
    assert [(int(v) >> 2) & 3 for v in t[0:8]] == [2] * 8  # weights 8..15: grid row 0, all +1 -> u = 2
    # out-of-range values are refused
    g_big = g3.copy(); g_big[7] = [17, 3, 5, 7]
    sb2 = np.zeros(102, np.uint8); sb2[2] = 7
    assert o.transcode_row(CB3, sb2, 256, g_big, CB3X)[1] == -1
    assert o.transcode_row(CB2, sb, 256, np.full((256, 8), 5, np.int8), CB2X)[1] == -1


# ------------------------------------------------------------------ grouping

def check_route_hand(o):
    ids = np.array([[5, 2, 7], [2, 0, 5]], np.int32)
    r = o.route_group(ids, 8)
    assert list(r["grp_expert"]) == [0, 2, 5, 7]
    assert list(r["grp_start"]) == [0, 1, 3, 5, 6] and r["n_groups"] == 4
    assert list(r["ent_src"]) == [1, 0, 1, 0, 1, 0], r["ent_src"]
    assert list(r["ent_dst"]) == [4, 1, 3, 0, 5, 2], r["ent_dst"]
    r = o.route_group(ids, 8, entry_base=10)
    assert list(r["grp_start"]) == [10, 11, 13, 15, 16]
    assert list(r["ent_src"][10:]) == [1, 0, 1, 0, 1, 0] and (r["ent_src"][:10] == -1).all()
    r = o.route_group(np.array([[3, 9, -1]], np.int32), 8)
    assert r["dropped"] == 2 and list(r["grp_expert"]) == [3] and list(r["grp_start"]) == [0, 1]


def check_route_invariants(o):
    rng = np.random.Generator(np.random.PCG64(17))
    for T, k, E in ((1, 2, 8), (4, 8, 64), (3, 8, 16), (4, 8, 128), (2, 6, 6)):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        base = int(rng.integers(0, 5))
        r = o.route_group(ids, E, entry_base=base)
        G, ge, gs = r["n_groups"], r["grp_expert"], r["grp_start"]
        assert G == len(np.unique(ids)) and list(ge) == sorted(set(ids.ravel().tolist()))
        assert gs[0] == base and gs[G] == base + T * k and (np.diff(gs) >= 1).all()
        assert (np.diff(gs) <= T).all()
        seen = set()
        for g in range(G):
            prev = -1
            for e in range(gs[g], gs[g + 1]):
                t, dst = r["ent_src"][e], r["ent_dst"][e]
                assert dst // k == t and ids[t, dst % k] == ge[g]
                assert dst > prev
                prev = dst
                seen.add(int(dst))
        assert seen == set(range(T * k))


# ------------------------------------------------------------------ grouped steps

def check_grouped_invariants(o):
    rng = np.random.Generator(np.random.PCG64(19))
    K, rows, E = 256, 24, 6
    for typ in (Q8_0, NL4, CB3):
        cb = _cb_for(typ, rng)
        blobs = [np.concatenate([_random_row(typ, K, rng) for _ in range(rows)]) for _ in range(E)]
        x = rng.standard_normal((5, K)).astype(np.float32)
        act = o.quantize_q8_1(x)
        ge = np.array([4, 1, 2], np.int32)
        gs = np.array([2, 4, 5, 8], np.int32)
        ent_in = np.array([-9, -9, 3, 0, 4, 1, 2, 0], np.int32)
        ent_out = np.array([-9, -9, 6, 1, 3, 0, 7, 2], np.int32)
        out = np.full((9, rows), np.nan)
        out, rc = o.grouped_gemv(typ, K, rows, blobs, ge, gs, 3, act, ent_in, ent_out, out, cb)
        assert rc == 0
        written = set()
        for g in range(3):
            for e in range(gs[g], gs[g + 1]):
                written.add(int(ent_out[e]))
                for r in (0, 7, rows - 1):
                    want = o.row_dot(typ, blobs[ge[g]][r * (len(blobs[0]) // rows):], K, act[ent_in[e]], cb)
                    assert out[ent_out[e], r] == want
        for i in range(9):
            assert np.isnan(out[i]).all() == (i not in written), "untouched rows"
        # permuting group order and renumbering entries leaves each entry's row unchanged
        perm = [2, 0, 1]
        ge2 = ge[perm]
        sizes = np.diff(gs)[perm]
        gs2 = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        src_e = np.concatenate([np.arange(gs[g], gs[g + 1]) for g in perm])
        out2 = np.full((9, rows), np.nan)
        out2, _ = o.grouped_gemv(typ, K, rows, blobs, ge2, gs2, 3, act, ent_in[src_e], ent_out[src_e], out2, cb)
        assert np.array_equal(np.isnan(out), np.isnan(out2))
        assert np.array_equal(out[~np.isnan(out)], out2[~np.isnan(out2)])
        # n_groups = 0 writes nothing; a bad expert id is reported and skipped
        out3 = np.full((9, rows), np.nan)
        o.grouped_gemv(typ, K, rows, blobs, ge, gs, 0, act, ent_in, ent_out, out3, cb)
        assert np.isnan(out3).all()
        _, rc = o.grouped_gemv(typ, K, rows, blobs, np.array([E, 1, 2], np.int32), gs, 3, act, ent_in, ent_out,
                               out3, cb)
        assert rc == -1 and np.isnan(out3[6]).all() and np.isnan(out3[1]).all()


def check_swiglu_q8_1(o):
    rng = np.random.Generator(np.random.PCG64(23))
    F = 64
    gu = (rng.standard_normal((6, 2 * F)) * 3).astype(np.float32)
    hq = np.full((6, F // 32, 36), 0xAB, np.uint8)
    o.swiglu_q8_1(gu, F, 2, 5, hq)
    assert (hq[:2] == 0xAB).all() and (hq[5:] == 0xAB).all(), "rows outside [e0, e1) untouched"
    for e in range(2, 5):
        h = o.swiglu(gu[e, :F], gu[e, F:])
        assert np.array_equal(hq[e], o.quantize_q8_1(h[None, :])[0])


# ------------------------------------------------------------------ router and combine

def check_router(o):
    ids, w, rc = o.router_topk(np.array([[0.5, 2, -1, 2, 3]], np.float32), 3)
    e = np.e
    assert rc == 0 and ids.tolist() == [[4, 1, 3]], ids
    assert np.allclose(w[0], [e / (e + 2), 1 / (e + 2), 1 / (e + 2)], rtol=0, atol=1e-15), w
    ids, w, rc = o.router_topk(np.full((2, 10), 0.25, np.float32), 4)
    assert rc == 0 and ids.tolist() == [[0, 1, 2, 3]] * 2 and np.allclose(w, 0.25, rtol=0, atol=1e-15)
    rng = np.random.Generator(np.random.PCG64(31))
    for E, k in ((8, 2), (64, 8), (128, 8), (40, 40)):
        lg = rng.standard_normal((5, E)).astype(np.float32)
        lg[0, 3] = lg[0, 7]  # a tie
        ids, w, rc = o.router_topk(lg, k)
        assert rc == 0
        for t in range(5):
            sel = list(ids[t])
            assert len(set(sel)) == k
            for a, b in zip(sel, sel[1:]):  # descending, ties by id
                assert lg[t, a] > lg[t, b] or (lg[t, a] == lg[t, b] and a < b)
            last = sel[-1]
            for x in range(E):
                if x not in sel:
                    assert lg[t, x] < lg[t, last] or (lg[t, x] == lg[t, last] and x > last)
            assert abs(w[t].sum() - 1.0) < 1e-12
            for j in range(1, k):
                assert abs(w[t, 0] / w[t, j] - np.exp(float(lg[t, sel[0]]) - float(lg[t, sel[j]]))) < 1e-9 * w[t, 0] / w[t, j]
    assert o.router_topk(np.zeros((1, 4), np.float32), 5)[2] == -1


def check_combine(o):
    rng = np.random.Generator(np.random.PCG64(37))
    T, k, E, N = 3, 4, 16, 64
    out = rng.standard_normal((T * k, N)).astype(np.float32)
    ids = np.tile(np.arange(k, dtype=np.int32), (T, 1))
    for j in range(k):  # one-hot weights read out row t*k + j
        w = np.zeros((T, k)); w[:, j] = 1.0
        y = o.combine(out, ids, w, E)
        assert np.array_equal(y, out[j::k].astype(np.float64))
    same = np.repeat(out[:T], k, axis=0)  # rows t*k .. t*k+k-1 all equal out[t]
    w = rng.random((T, k))
    y = o.combine(same, ids, w, E)
    assert np.allclose(y, out[:T].astype(np.float64) * w.sum(1, keepdims=True), rtol=1e-14, atol=0)
    # hand-worked: 2 tokens, k = 2, N = 2
    o2 = np.array([[1, 2], [3, 4], [5, 6], [7, 8]], np.float32)
    y = o.combine(o2, np.array([[0, 1], [2, 3]], np.int32), np.array([[0.25, 0.75], [0.5, 0.5]]), 4)
    assert y.tolist() == [[2.5, 3.5], [6.0, 7.0]], y
    # a dropped id (outside [0, E)) contributes nothing
    y = o.combine(o2, np.array([[0, -1], [9, 3]], np.int32), np.array([[0.25, 0.75], [0.5, 0.5]]), 4)
    assert y.tolist() == [[0.25, 0.5], [3.5, 4.0]], y


# ------------------------------------------------------------------ QSA block scores

def check_qsa_hand(o):
    """Hand-worked blocks, one per case, each key nonzero only in its own dims (so the queries'
    other values meet zeros: q*0 and fma(q, 0, p) = p are exact, and the pairings add zeros):
      block 0: lane 0 takes dims 0..3 and fuses its products: q0*k0 = -3, then fma((1 + 2^-23), 3,
               -3) = 3 * 2^-23 exactly (a rounded product first would give 3 + 2^-21 - 3 = 2^-21)
      block 1: dims 4, 5, 6 sit in one lane (1): 2^-24, then 2^-23, then 1 + 2^-23 exactly (in three
               lanes the pairings would add 1 + 2^-24 first, which rounds to 1)
      block 2: lanes 2, 3 and 19 hold 2^24, 1, 1: level 16 pairs lanes 3 and 19 (2), level 1 adds
               2^24 + 2 = 16777218 exactly (a sum in lane order loses both ones: 16777216)
      block 3: one dim, heads give relus 1, 2^-24, 2^-24, 0: head order ((1 + 2^-24) + 2^-24) + 0
               = 1 (in reverse order 1 + 2^-23)
      block 4: scale 4; head 0's dot -6 is dropped by the relu, head 1's 1.5 * 4 = 6
      block 5: the tail, zero key: 0 + 1e9"""
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
    got = o.qsa_block_scores(q, keys, scale)[0]
    want = np.array([3 * 2.0 ** -23, 1 + 2.0 ** -23, 16777218.0, 1.0, 6.0, 1e9], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (got, want)


def check_qsa_bruteforce(o):
    """Random queries, keys and scales against the fp64 definition sum_h max(scale * q_h . k, 0)
    (+ 1e9 on the tail): every fp32 result within 16 * 2^-24 of scale * sum_h sum_d |q_hd k_d| (a
    bound on 4 in-lane steps, 5 pairing levels, the scale product and 3 head additions), plus
    half an ulp of 1e9 on the tail; and each query's and each non-tail block's scores depend on
    nothing else (the same bits alone and among others)."""
    rng = np.random.Generator(np.random.PCG64(11))
    T, nb = 4, 37
    q = rng.standard_normal((T, 4, 128)).astype(np.float32)
    keys = rng.integers(-127, 128, (nb, 128)).astype(np.int8)
    scale = rng.uniform(1e-3, 1e-2, nb).astype(np.float32)
    got = o.qsa_block_scores(q, keys, scale)
    qk = np.einsum("thd,bd->thb", q.astype(np.float64), keys.astype(np.float64)) * scale.astype(np.float64)
    ref = np.maximum(qk, 0.0).sum(axis=1)
    mag = (np.einsum("thd,bd->tb", np.abs(q.astype(np.float64)), np.abs(keys.astype(np.float64)))
           * scale.astype(np.float64))
    ref[:, -1] += 1e9
    bound = 16 * 2.0 ** -24 * mag
    bound[:, -1] += 32.0
    assert (np.abs(got.astype(np.float64) - ref) <= bound).all()
    assert (got[:, :-1] >= 0).all()
    # independence: one query alone, and the non-tail blocks in another order with another tail
    assert np.array_equal(o.qsa_block_scores(q[2:3], keys, scale)[0].view(np.uint32), got[2].view(np.uint32))
    perm = rng.permutation(nb - 1)
    keys2 = np.concatenate([keys[:-1][perm], keys[-1:]])
    sc2 = np.concatenate([scale[:-1][perm], scale[-1:]])
    got2 = o.qsa_block_scores(q, keys2, sc2)
    assert np.array_equal(got2[:, :-1].view(np.uint32), got[:, :-1][:, perm].view(np.uint32))


ALL_CHECKS = [check_qsa_hand, check_qsa_bruteforce, check_router, check_combine, check_f16, check_exp, check_silu, check_q8_1, check_formats_hand, check_formats_onehot,
              check_formats_bruteforce, check_slots, check_route_hand, check_route_invariants, check_grouped_invariants,
              check_swiglu_q8_1]
