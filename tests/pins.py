"""Pins of the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` takes an ``oracle.OracleLib`` and raises AssertionError when the
oracle disagrees with:
  * hand-worked fixtures (tests/golden/hand_worked.json),
  * the independent pure-Python brute force (oracle/brute.py), on random tiny
    cases and an exhaustive sweep,
  * the routing invariants, which together determine the stable permutation
    uniquely (so they are a complete, independent specification),
  * closed forms (identity routing, one expert, K = 1 equals a stable library
    argsort),
  * torch's fp32 -> bf16 conversion (an independent round-to-nearest-even),
  * an fp64 recomputation of unpermute within the fp32-accumulation plus
    bf16-rounding error bound.
The same functions are run against deliberately broken copies of the oracle
(tests/test_oracle_mutants.py) to show that plausible mistakes are caught.

Definitions: vLLM PR #14568 description (permute / unpermute semantics) and
vLLM PR #43014 digest, "key source excerpts" (buffer shapes and dtypes).
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
import torch

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "hand_worked.json")


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------- helpers ---

def local_keys(topk_ids, E, expert_map=None, E_local=None):
    """Local expert per expanded row (-1 = dropped), vectorised numpy."""
    g = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    valid = (g >= 0) & (g < E)
    keys = np.full(g.shape, -1, np.int64)
    if expert_map is None:
        keys[valid] = g[valid]
    else:
        m = np.asarray(expert_map, dtype=np.int64)
        e = m[g[valid]]
        e_ok = (e >= 0) & (e < (E_local if E_local is not None else E))
        keys[np.flatnonzero(valid)[e_ok]] = e[e_ok]
    return keys


def check_routing_invariants(topk_ids, E, res, expert_map=None, E_local=None):
    """Routing invariants.  Together they determine the stable sort uniquely:
    segment sizes = per-expert counts, p -> r a bijection onto the valid rows,
    keys constant on each segment, r strictly increasing inside a segment."""
    E_local = E if E_local is None else E_local
    keys = local_keys(topk_ids, E, expert_map, E_local)
    R = keys.shape[0]
    off = np.asarray(res["offsets"], dtype=np.int64)
    pidx = np.asarray(res["permuted_idx"], dtype=np.int64)
    inv = np.asarray(res["inv_permuted_idx"], dtype=np.int64)
    assert off.shape == (E_local + 1,)
    assert pidx.shape == (R,) and inv.shape == (R,)
    counts = np.bincount(keys[keys >= 0], minlength=E_local)
    assert off[0] == 0
    assert np.all(np.diff(off) == counts), "segment sizes != expert counts"
    n_valid = int(counts.sum())
    assert off[-1] == n_valid
    assert np.all(pidx[n_valid:] == -1), "tail of permuted_idx must be -1"
    assert np.all(inv[keys < 0] == -1), "dropped rows must have inv -1"
    head = pidx[:n_valid]
    assert np.all((head >= 0) & (head < R))
    assert np.all(keys[head] >= 0), "a dropped row was placed"
    assert np.all(inv[head] == np.arange(n_valid)), "inv o permuted_idx != id"
    assert np.unique(head).shape[0] == n_valid, "a row appears twice"
    seg = np.repeat(np.arange(E_local), counts)
    assert np.all(keys[head] == seg), "row placed in the wrong expert segment"
    if n_valid > 1:
        same = seg[1:] == seg[:-1]
        assert np.all(head[1:][same] > head[:-1][same]), "order not stable"


def bf16_bits_to_f64(bits):
    u = np.asarray(bits, dtype=np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_bits_exact(vals):
    """Bits of values that are exactly representable in bf16."""
    f = np.asarray(vals, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "fixture value is not exact in bf16"
    return (u >> 16).astype(np.uint16)


def torch_bf16_bits(x_f32):
    t = torch.from_numpy(np.asarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def random_tiny_routing(rng, T, K, E, with_map, allow_bad):
    lo, hi = (-1, E + 1) if allow_bad else (0, E)
    ids = rng.integers(lo, hi, size=(T, K))
    emap = None
    E_local = E
    if with_map:
        E_local = int(rng.integers(1, E + 1))
        emap = np.full(E, -1, np.int32)
        chosen = rng.choice(E, size=E_local, replace=False)
        emap[chosen] = rng.permutation(E_local)
        if allow_bad and rng.random() < 0.3:
            emap[int(rng.integers(0, E))] = E_local  # out of local range
    return ids, emap, E_local


def brute_equal(res, ref):
    assert list(np.asarray(res["offsets"])) == list(ref["offsets"])
    assert list(np.asarray(res["permuted_idx"])) == list(ref["permuted_idx"])
    assert list(np.asarray(res["inv_permuted_idx"])) == list(ref["inv_permuted_idx"])
    assert res["flags"] == ref["flags"]


# ------------------------------------------------------------------- pins ---

def pin_golden_routing(orc):
    for case in load_golden()["routing"]:
        ids = np.array(case["topk_ids"], np.int32)
        emap = None if case["expert_map"] is None else np.array(case["expert_map"], np.int32)
        res = orc.permute(ids, case["E"], expert_map=emap, E_local=case["E_local"])
        assert list(res["offsets"]) == case["offsets"], case["name"]
        assert list(res["permuted_idx"]) == case["permuted_idx"], case["name"]
        assert list(res["inv_permuted_idx"]) == case["inv_permuted_idx"], case["name"]
        assert res["flags"] == case["flags"], case["name"]


def pin_golden_unpermute(orc):
    for case in load_golden()["unpermute"]:
        rows = f64_to_bf16_bits_exact(case["rows"])
        if "topk_weights_f32_bits" in case:
            w = np.array(case["topk_weights_f32_bits"], np.uint32).view(np.float32)
        else:
            w = np.array(case["topk_weights"], np.float32)
        inv = np.array(case["inv_permuted_idx"], np.int32)
        out, flags = orc.unpermute(rows, w, inv)
        assert flags == case.get("flags", 0), case["name"]
        assert out.tolist() == case["out_bf16_bits"], case["name"]
        if "out" in case:
            assert bf16_bits_to_f64(out).tolist() == case["out"], case["name"]


def pin_golden_rounding(orc):
    g = load_golden()["rounding"]
    x = np.array(g["f32_bits"], np.uint32).view(np.float32)
    assert orc.f32_to_bf16_rne(x).tolist() == g["bf16_bits"]


def pin_rounding_vs_torch(orc, n=200000, seed=1):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    # force many exact ties and near-ties, odd and even kept halves
    bits[: n // 4] = (bits[: n // 4] & 0xFFFF0000) | 0x8000
    bits[n // 4: n // 2] = (bits[n // 4: n // 2] & 0xFFFF0000) | rng.choice(
        np.array([0x7FFF, 0x8001, 0xFFFF, 0x0001], np.uint32), size=n // 2 - n // 4)
    x = bits.view(np.float32)
    nan = np.isnan(x)
    got = orc.f32_to_bf16_rne(x)
    want = torch_bf16_bits(x)
    assert np.array_equal(got[~nan], want[~nan])
    # NaN stays NaN (quiet), sign kept
    g = got[nan].astype(np.uint32)
    assert np.all(((g & 0x7F80) == 0x7F80) & ((g & 0x007F) != 0))
    assert np.array_equal(g >> 15, (bits[nan] >> 31))


def pin_brute_random(orc, n_cases=300, seed=2):
    rng = np.random.default_rng(seed)
    for _ in range(n_cases):
        T = int(rng.integers(0, 13))
        K = int(rng.integers(1, 4))
        E = int(rng.integers(1, 7))
        with_map = bool(rng.random() < 0.5)
        ids, emap, E_local = random_tiny_routing(rng, T, K, E, with_map, True)
        for dt in (np.int32, np.int64):
            res = orc.permute(ids.astype(dt).reshape(T, K), E, expert_map=emap,
                              E_local=E_local)
            ref = brute.permute(ids.tolist(), E, expert_map=emap, E_local=E_local)
            brute_equal(res, ref)
        # unpermute on the same routing with random bf16 rows and fp32 weights
        H = int(rng.integers(1, 5))
        R = T * K
        if R == 0:
            continue
        rows_f = rng.standard_normal((R, H)).astype(np.float32)
        rows = torch_bf16_bits(rows_f)
        w = rng.random((T, K)).astype(np.float32)
        inv = np.array(brute.permute(ids.tolist(), E, expert_map=emap,
                                     E_local=E_local)["inv_permuted_idx"], np.int32)
        out, _ = orc.unpermute(rows, w, inv)
        sums = brute.unpermute_f32_sums(bf16_bits_to_f64(rows).tolist(),
                                        w.astype(np.float64).tolist(), inv.tolist(),
                                        T, K, H)
        want = torch_bf16_bits(np.array(sums, np.float32).reshape(T, H))
        assert np.array_equal(out, want)


def pin_exhaustive_tiny(orc):
    """Every assignment of ids in {-1..4} for T<=2, K=2, E=4 and every
    assignment in {0..3} for T=3, K=2, with and without an expert map."""
    E = 4
    maps = [None, np.array([1, -1, 0, -1], np.int32)]
    cases = []
    for T, values in ((1, range(-1, 5)), (2, range(-1, 5)), (3, range(0, 4))):
        for flat in itertools.product(values, repeat=T * 2):
            cases.append(np.array(flat, np.int32).reshape(T, 2))
    for emap in maps:
        E_local = E if emap is None else 2
        for ids in cases:
            res = orc.permute(ids, E, expert_map=emap, E_local=E_local)
            ref = brute.permute(ids.tolist(), E, expert_map=emap, E_local=E_local)
            brute_equal(res, ref)


def pin_invariants(orc, seed=3):
    rng = np.random.default_rng(seed)
    for T, K, E, with_map in ((1, 1, 1, False), (257, 8, 128, False),
                              (1000, 6, 64, True), (64, 8, 256, False),
                              (333, 2, 8, True)):
        ids, emap, E_local = random_tiny_routing(rng, T, K, E, with_map, False)
        # skew: half the rows hit expert 0
        ids[rng.random(ids.shape) < 0.5] = 0
        res = orc.permute(ids.astype(np.int32), E, expert_map=emap, E_local=E_local)
        check_routing_invariants(ids, E, res, emap, E_local)
        res64 = orc.permute(ids.astype(np.int64), E, expert_map=emap, E_local=E_local)
        for key in ("offsets", "permuted_idx", "inv_permuted_idx"):
            assert np.array_equal(res[key], res64[key])


def pin_closed_forms(orc, seed=4):
    rng = np.random.default_rng(seed)
    # identity: K = 1 and non-decreasing ids -> the identity permutation
    T, E = 37, 5
    ids = np.sort(rng.integers(0, E, size=T)).reshape(T, 1).astype(np.int32)
    res = orc.permute(ids, E)
    assert np.array_equal(res["permuted_idx"], np.arange(T))
    assert np.array_equal(res["inv_permuted_idx"], np.arange(T))
    # every row on one expert j: offsets = [0]*(j+1) + [R]*(E-j); order = r
    T, K, E, j = 9, 3, 6, 4
    res = orc.permute(np.full((T, K), j, np.int32), E)
    R = T * K
    assert res["offsets"].tolist() == [0] * (j + 1) + [R] * (E - j)
    assert np.array_equal(res["permuted_idx"], np.arange(R))
    # K = 1: the permutation is the stable argsort of the ids
    T, E = 500, 16
    ids = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    res = orc.permute(ids, E)
    assert np.array_equal(res["permuted_idx"], np.argsort(ids[:, 0], kind="stable"))
    # expanded ids: stable argsort of the flattened [T,K] ids, for any K
    T, K, E = 300, 4, 8
    ids = rng.integers(0, E, size=(T, K)).astype(np.int32)
    res = orc.permute(ids, E)
    assert np.array_equal(res["permuted_idx"], np.argsort(ids.reshape(-1), kind="stable"))
    # T = 0
    res = orc.permute(np.zeros((0, 4), np.int32), 8)
    assert res["offsets"].tolist() == [0] * 9


def pin_rows_copied(orc, seed=5):
    rng = np.random.default_rng(seed)
    T, K, E, H = 50, 4, 8, 96
    ids, emap, E_local = random_tiny_routing(rng, T, K, E, True, False)
    for dt in (np.uint16, np.uint8):  # bf16 bits and fp8 bytes
        hidden = rng.integers(0, np.iinfo(dt).max, size=(T, H), dtype=dt)
        scales = rng.random((T, H // 32)).astype(np.float32)
        res = orc.permute(ids.astype(np.int32), E, expert_map=emap, E_local=E_local,
                          hidden=hidden, scales=scales)
        n = res["n_valid"]
        src = res["permuted_idx"][:n] // K
        assert np.array_equal(res["permuted_hidden"][:n], hidden[src])
        assert np.array_equal(res["permuted_scales"][:n], scales[src])
        # untouched tail: the marshalling zero-fills it and the oracle never writes it
        assert not res["permuted_hidden"][n:].any()


def pin_unpermute_one_hot(orc, seed=6):
    rng = np.random.default_rng(seed)
    T, K, H = 40, 6, 64
    rows = torch_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    inv = rng.permutation(T * K).astype(np.int32)
    hot = rng.integers(0, K, size=T)
    w = np.zeros((T, K), np.float32)
    w[np.arange(T), hot] = 1.0
    out, _ = orc.unpermute(rows, w, inv)
    want = rows[inv.reshape(T, K)[np.arange(T), hot]]
    assert np.array_equal(out, want)
    # round trip: identical rows with weights summing to 1 return x within 1 ulp
    x = rng.standard_normal((T, H)).astype(np.float32)
    xb = torch_bf16_bits(x)
    rows = np.repeat(xb, K, axis=0)  # rows of token t at t*K..t*K+K-1
    w = rng.random((T, K)).astype(np.float32)
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    out, _ = orc.unpermute(rows, w, np.arange(T * K, dtype=np.int32))
    got = bf16_bits_to_f64(out)
    ref = bf16_bits_to_f64(xb)
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)


def pin_unpermute_bound(orc, seed=7):
    """fp64 sum vs oracle: |out - exact| <= 2^-8 |exact| + 1.01 K 2^-24 sum|w x|
    (bf16 rounding of an fp32 sum whose own error is at most K u32 sum|w x|)."""
    rng = np.random.default_rng(seed)
    T, K, H = 64, 8, 256
    R = T * K
    rows = torch_bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    w = rng.random((T, K)).astype(np.float32)
    inv = rng.permutation(R).astype(np.int32)
    inv[rng.random(R) < 0.2] = -1
    out, _ = orc.unpermute(rows, w, inv)
    x = bf16_bits_to_f64(rows)
    invm = inv.reshape(T, K)
    gathered = np.where((invm >= 0)[:, :, None], x[np.maximum(invm, 0)], 0.0)
    terms = w.astype(np.float64)[:, :, None] * gathered
    exact = terms.sum(axis=1)
    mag = np.abs(terms).sum(axis=1)
    bound = 2.0 ** -8 * np.abs(exact) + 1.01 * K * 2.0 ** -24 * mag * (1 + 2.0 ** -7) + 1e-37
    err = np.abs(bf16_bits_to_f64(out) - exact)
    assert np.all(err <= bound), float((err - bound).max())


def pin_flags(orc):
    ids = np.array([[0, 5], [1, 2]], np.int32)
    assert orc.permute(ids, 5)["flags"] == 1
    emap = np.array([0, -1, 7, 1, -1], np.int32)
    assert orc.permute(np.array([[0, 2]], np.int32), 5, expert_map=emap, E_local=2)["flags"] == 2
    assert orc.permute(np.array([[0, 1]], np.int32), 5, expert_map=emap, E_local=2)["flags"] == 0
    rows = np.zeros((2, 3), np.uint16)
    _, f = orc.unpermute(rows, np.ones((1, 2), np.float32), np.array([0, 2], np.int32))
    assert f == 4
    # below -1 names no row either; -1 itself is a dropped row, not an error
    _, f = orc.unpermute(rows, np.ones((1, 2), np.float32), np.array([-2, 1], np.int32))
    assert f == 4
    _, f = orc.unpermute(rows, np.ones((1, 2), np.float32), np.array([-1, 1], np.int32))
    assert f == 0


# ------------------------------------------------------ fp8 quantisation ---

def e4m3_value(c):
    """Value of one e4m3 ("fn") code, from the format: sign, 4-bit exponent
    (bias 7), 3-bit mantissa; exponent 0 is subnormal; 0x7F / 0xFF are NaN."""
    sign = -1.0 if c & 0x80 else 1.0
    e = (c >> 3) & 0xF
    m = c & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def pin_e4m3_exhaustive(orc):
    """Every finite code decodes and re-encodes to itself (signed zero kept)."""
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    vals = np.array([e4m3_value(c) for c in codes], np.float64)
    x = vals.astype(np.float32)
    assert np.array_equal(x.astype(np.float64), vals)  # all exact in fp32
    x[codes.index(0x80)] = np.float32(-0.0)
    got = orc.f32_to_e4m3(x)
    assert got.tolist() == codes


def pin_e4m3_ties_and_neighbours(orc):
    """Midpoints between neighbouring finite values go to the even code;
    points just off a midpoint go to the nearer code."""
    pos = [c for c in range(0x7F) if c != 0x7F]
    for c in pos[:-1]:
        lo, hi = e4m3_value(c), e4m3_value(c + 1)
        mid = (lo + hi) / 2.0
        even = c if (c & 1) == 0 else c + 1
        x = np.array([mid, np.nextafter(np.float32(mid), np.float32(0)),
                      np.nextafter(np.float32(mid), np.float32(1e9))], np.float32)
        assert float(x[0]) == mid
        got = orc.f32_to_e4m3(x).tolist()
        assert got == [even, c, c + 1], (c, got)
        neg = orc.f32_to_e4m3(-x).tolist()
        assert neg == [even | 0x80, c | 0x80, (c + 1) | 0x80]


def pin_e4m3_vs_torch_and_saturation(orc, seed=8):
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.standard_normal(100000) * 50, rng.uniform(-448, 448, 100000),
                        rng.standard_normal(50000) * 1e-3]).astype(np.float32)
    got = orc.f32_to_e4m3(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)
    big = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, np.inf], np.float32)
    assert orc.f32_to_e4m3(big).tolist() == [0x7E] * 7
    assert orc.f32_to_e4m3(-big).tolist() == [0xFE] * 7
    nan = orc.f32_to_e4m3(np.array([np.nan, -np.nan], np.float32)).tolist()
    assert [c & 0x7F for c in nan] == [0x7F, 0x7F]


def pin_quantize_golden(orc):
    g = load_golden()["quantize_fp8"]
    G = g["group"]
    groups = g["groups"]
    x = np.zeros((1, G * len(groups)), np.float32)
    for gi, grp in enumerate(groups):
        for i, v in grp["nonzero"].items():
            x[0, gi * G + int(i)] = v
    bits = f64_to_bf16_bits_exact(x)
    codes, scales = orc.quantize_fp8(bits, G)
    for gi, grp in enumerate(groups):
        want = np.zeros(G, np.uint8)
        for i, c in grp["codes_nonzero"].items():
            want[int(i)] = c
        assert codes[0, gi * G:(gi + 1) * G].tolist() == want.tolist(), grp["name"]
        expr = grp["scale_is"]
        if expr == "1":
            assert scales[0, gi] == np.float32(1.0)
        else:
            num = float(expr.split("fp32(")[1].split(")")[0])
            assert scales[0, gi] == np.float32(num) / np.float32(448.0), grp["name"]


def pin_quantize_properties(orc, seed=9):
    rng = np.random.default_rng(seed)
    T, H, G = 37, 512, 128
    x = rng.standard_normal((T, H)).astype(np.float32) * rng.uniform(0.01, 100, (T, 1)).astype(np.float32)
    x[3, 128:256] = 0.0  # an all-zero group
    bits = torch_bf16_bits(x)
    xb = bf16_bits_to_f64(bits)
    codes, scales = orc.quantize_fp8(bits, G)
    vals = np.vectorize(e4m3_value)(codes.astype(np.int64))
    deq = vals * np.repeat(scales.astype(np.float64), G, axis=1)
    amax = np.abs(xb).reshape(T, H // G, G).max(axis=2)
    nz = amax > 0
    assert np.all(scales[~nz] == 1.0) and np.all(codes.reshape(T, H // G, G)[~nz] == 0)
    assert np.array_equal(scales[nz], (amax[nz].astype(np.float32) / np.float32(448.0)))
    top = np.abs(vals).reshape(T, H // G, G).max(axis=2)
    assert np.all(top[nz] == 448.0)
    s = np.repeat(scales.astype(np.float64), G, axis=1)
    # half an e4m3 ulp (2^-4 relative) of the scaled value, or half the
    # subnormal step (2^-10 * scale), plus the fp32 division's own rounding
    bound = np.maximum(np.abs(xb) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(np.abs(deq - xb) <= bound)


# -------------------------------------------------------- batched layout ---

def pin_batched_golden(orc):
    for c in load_golden()["batched"]:
        emap = None if c["expert_map"] is None else np.array(c["expert_map"], np.int32)
        r = orc.permute_batched(np.array(c["topk_ids"], np.int32), c["E"], c["M"],
                                expert_map=emap, E_local=c["E_local"])
        assert r["expert_num_tokens"].tolist() == c["expert_num_tokens"], c["name"]
        assert r["inv_permuted_idx"].tolist() == c["inv_permuted_idx"], c["name"]
        assert r["flags"] == c["flags"], c["name"]


def pin_batched_brute_random(orc, n_cases=200, seed=10):
    rng = np.random.default_rng(seed)
    for _ in range(n_cases):
        T = int(rng.integers(0, 12))
        K = int(rng.integers(1, 4))
        E = int(rng.integers(1, 6))
        M = int(rng.integers(1, 6))  # small capacities: overflow is common
        ids, emap, E_local = random_tiny_routing(rng, T, K, E, bool(rng.random() < 0.5), True)
        res = orc.permute_batched(ids.astype(np.int32).reshape(T, K), E, M, expert_map=emap,
                                  E_local=E_local)
        ref = brute.permute_batched(ids.tolist(), E, M, expert_map=emap, E_local=E_local)
        assert res["expert_num_tokens"].tolist() == ref["expert_num_tokens"]
        assert res["inv_permuted_idx"].tolist() == ref["inv_permuted_idx"]
        assert res["flags"] == ref["flags"]


def pin_batched_vs_contiguous(orc, seed=11):
    """With room for every row, slot = e*M + (p - offset[e]) where p is the
    row's position in the contiguous layout, and each slot holds its token."""
    rng = np.random.default_rng(seed)
    T, K, E, H = 200, 6, 16, 24
    ids, emap, E_local = random_tiny_routing(rng, T, K, E, True, False)
    hidden = rng.integers(0, 65535, size=(T, H), dtype=np.uint16)
    cont = orc.permute(ids.astype(np.int32), E, expert_map=emap, E_local=E_local)
    M = int(np.diff(cont["offsets"]).max()) + 3
    bat = orc.permute_batched(ids.astype(np.int32), E, M, expert_map=emap, E_local=E_local,
                              hidden=hidden)
    assert bat["flags"] == 0
    assert np.array_equal(bat["expert_num_tokens"], np.diff(cont["offsets"]))
    inv_c = cont["inv_permuted_idx"]
    keys = local_keys(ids, E, emap, E_local)
    want = np.where(inv_c >= 0, keys * M + (inv_c - cont["offsets"][np.maximum(keys, 0)]), -1)
    assert np.array_equal(bat["inv_permuted_idx"], want)
    slots = bat["inv_permuted_idx"][bat["inv_permuted_idx"] >= 0]
    rows = np.flatnonzero(bat["inv_permuted_idx"] >= 0)
    assert np.array_equal(bat["batched_hidden"][slots], hidden[rows // K])


ALL_PINS = [pin_golden_routing, pin_golden_unpermute, pin_golden_rounding,
            pin_rounding_vs_torch, pin_brute_random, pin_exhaustive_tiny,
            pin_invariants, pin_closed_forms, pin_rows_copied,
            pin_unpermute_one_hot, pin_unpermute_bound, pin_flags,
            pin_e4m3_exhaustive, pin_e4m3_ties_and_neighbours,
            pin_e4m3_vs_torch_and_saturation, pin_quantize_golden, pin_quantize_properties,
            pin_batched_golden, pin_batched_brute_random, pin_batched_vs_contiguous]
