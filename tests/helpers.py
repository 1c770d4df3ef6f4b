"""Comparison helpers shared by the GPU parity tests.

Tolerances (floating point, bf16 storage with fp32 accumulation):
  * elementwise |gpu - oracle| <= max(2e-2, one bf16 spacing at the oracle
    value).  2e-2 is the required bound; where a bf16 step itself exceeds it
    (|v| >= 4, step >= 2^-5), two correct roundings of nearly equal sums can
    land one step apart, so the bound there is that one step.
  * relative L2 over the tensor <= 1e-2.
Router logits are float32 sums of K bf16 products: compared with an absolute
bound of 1e-3 (fp32 accumulation error of a length-K dot product with the
workloads' magnitudes is ~1e-5).
"""
from __future__ import annotations

import numpy as np

import oracle as O

ATOL = 2e-2
REL_L2 = 1e-2
LOGIT_ATOL = 1e-3


def bf16_step(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (2^(e-8) in the binade [2^(e-1), 2^e))."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))
    return np.ldexp(1.0, e - 8)


def check_close(name: str, got, want, report: dict | None = None):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = np.abs(got - want)
    bound = np.maximum(ATOL, bf16_step(want))
    worst = float((err / bound).max()) if err.size else 0.0
    nrm = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(got - want) / nrm) if nrm > 0 else float(np.linalg.norm(got))
    if report is not None:
        report[name] = {"max_abs": float(err.max()) if err.size else 0.0, "rel_l2": rel,
                        "n_over_atol": int((err > ATOL).sum())}
    assert worst <= 1.0, f"{name}: max abs err {err.max():.4g} exceeds bound (ratio {worst:.3g})"
    assert rel <= REL_L2, f"{name}: relative L2 {rel:.3g} > {REL_L2}"


def tie_margin_ok(logits32: np.ndarray, k: int, idx_o: np.ndarray, slack: float):
    """Tokens whose oracle gaps (adjacent top-(k+1) logits) all sit more than
    `slack` away from the near-tie threshold, so the flag cannot flip.  With
    logits that differ by at most err, a gap moves by at most 2*err: callers
    pass slack = 2*err (plus a hair)."""
    l = logits32.astype(np.float64)
    order = np.argsort(-l, axis=1, kind="stable")[:, : min(k + 1, l.shape[1])]
    top = np.take_along_axis(l, order, axis=1)
    gaps = top[:, :-1] - top[:, 1:]
    return (np.abs(gaps - O.TIE_EPS) > slack).all(axis=1)


def dispatch_rules_hold(idx: np.ndarray, slot_of, drop, expert_rows, count, plan):
    """Property check of a dispatch result against the rules, for the
    routing it was given: sender slots are ranks in priority order within
    (src, dst, wave) capped at c_send, receiver rows ranks within the
    expert over sender-kept rows capped at c_recv, rows laid out
    destination-major.  Used when near-ties make the GPU's routing differ
    from the oracle's in a few tokens."""
    T, k = idx.shape
    p = plan
    seen_key = {}
    seen_e = {}
    rows_e = {}
    for t in range(T):
        s = t // p.T_s
        for j in range(k):
            e = int(idx[t, j])
            dst, q = e // p.E_l, e % p.E_l
            wv = q // p.E_w
            key = (s, dst, wv)
            n = seen_key.get(key, 0)
            seen_key[key] = n + 1
            if n >= p.c_send:
                assert drop[t, j] == O.DROP_SEND and slot_of[t, j] == -1, (t, j)
                continue
            row = ((dst * p.W + wv) * p.S + s) * p.c_send + n
            r = seen_e.get(e, 0)
            seen_e[e] = r + 1
            if r >= p.c_recv:
                assert drop[t, j] == O.DROP_RECV and slot_of[t, j] == -1, (t, j)
                continue
            assert drop[t, j] == O.DROP_KEPT and slot_of[t, j] == row, (t, j)
            rows_e.setdefault(e, []).append(row)
    for e in range(p.E):
        rr = rows_e.get(e, [])
        assert count[e] == len(rr)
        assert list(expert_rows[e, : len(rr)]) == rr
        assert (expert_rows[e, len(rr):] == -1).all()


def ragged_rules_hold(idx: np.ndarray, slot_of, expert_offsets, expert_rows, count, plan):
    """Property check of a dropless ragged dispatch for the routing it was
    given: the pool is a permutation of 0..T*k-1 ordered by (destination,
    wave, source) blocks in priority order, and each expert's list holds its
    rows in priority order."""
    T, k = idx.shape
    p = plan
    keys = []
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            dst, q = e // p.E_l, e % p.E_l
            keys.append(((dst, q // p.E_w, t // p.T_s), t, j))
    for r, (_, t, j) in enumerate(sorted(keys)):
        assert slot_of[t, j] == r, (t, j)
    per = {}
    for t in range(T):
        for j in range(k):
            per.setdefault(int(idx[t, j]), []).append(int(slot_of[t, j]))
    for e in range(p.E):
        rows = per.get(e, [])
        assert count[e] == len(rows)
        assert list(expert_rows[expert_offsets[e]:expert_offsets[e + 1]]) == rows
