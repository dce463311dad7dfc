"""Pure-Python brute force for tiny inputs, written independently of the C oracle.

TEST INFRASTRUCTURE ONLY (used by the oracle's pin tests).  It restates the
definition as directly as Python allows: the permutation is Python's stable
``sorted`` of the valid expanded rows r = t*K + k keyed by local expert, and
unpermute is a literal double loop.  It must only ever run on tiny inputs.

Definitions: vLLM PR #14568 description (permute orders the expanded tokens by
expert; unpermute reduces them with the top-k weights) and the vLLM PR #43014
digest, "key source excerpts" (buffer shapes and dtypes).
"""
from __future__ import annotations

import struct


def local_expert(g: int, E: int, expert_map, E_local: int):
    """(local expert or None, flag) for one global id."""
    if g < 0 or g >= E:
        return None, 1
    if expert_map is None:
        return g, 0
    e = int(expert_map[g])
    if e == -1:
        return None, 0
    if e < 0 or e >= E_local:
        return None, 2
    return e, 0


def permute(topk_ids, E, expert_map=None, E_local=None):
    """topk_ids: list of lists [T][K] of Python ints."""
    T = len(topk_ids)
    K = len(topk_ids[0]) if T else 0
    if E_local is None:
        E_local = E
    keys = {}
    flags = 0
    for t in range(T):
        for k in range(K):
            e, f = local_expert(int(topk_ids[t][k]), E, expert_map, E_local)
            flags |= f
            if e is not None:
                keys[t * K + k] = e
    order = sorted(keys, key=lambda r: keys[r])  # stable: ties keep r order
    R = T * K
    permuted_idx = order + [-1] * (R - len(order))
    inv = [-1] * R
    for p, r in enumerate(order):
        inv[r] = p
    offsets = [sum(1 for r in keys if keys[r] < e) for e in range(E_local + 1)]
    return dict(offsets=offsets, permuted_idx=permuted_idx, inv_permuted_idx=inv,
                n_valid=len(order), flags=flags)


def _f32(x: float) -> float:
    """Round a Python float (binary64) to the nearest binary32."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def unpermute_f32_sums(rows, w, inv, T, K, H):
    """fp32 sums before the final rounding: acc = fl32(acc + fl32(w*x)), k ascending.

    rows: list of lists of Python floats (already exact bf16 values).
    Returns a [T][H] list of binary32 values held in Python floats.
    """
    out = []
    for t in range(T):
        line = []
        for h in range(H):
            acc = 0.0
            for k in range(K):
                p = inv[t * K + k]
                if p < 0 or p >= len(rows):
                    continue
                acc = _f32(acc + _f32(_f32(w[t][k]) * rows[p][h]))
            line.append(acc)
        out.append(line)
    return out


def permute_batched(topk_ids, E, M, expert_map=None, E_local=None):
    """Batched layout by the definition: the k-th row (in r order) routed to
    local expert e lands in slot e*M + k if k < M, else it is dropped."""
    T = len(topk_ids)
    K = len(topk_ids[0]) if T else 0
    if E_local is None:
        E_local = E
    placed = {e: [] for e in range(E_local)}
    inv = [-1] * (T * K)
    flags = 0
    for t in range(T):
        for k in range(K):
            r = t * K + k
            e, f = local_expert(int(topk_ids[t][k]), E, expert_map, E_local)
            flags |= f
            if e is None:
                continue
            if len(placed[e]) >= M:
                flags |= 16
                placed[e].append(None)
                continue
            inv[r] = e * M + len(placed[e])
            placed[e].append(r)
    counts = [min(len(placed[e]), M) for e in range(E_local)]
    return dict(expert_num_tokens=counts, inv_permuted_idx=inv, flags=flags)
