"""Plain float64 statement of the pooled-wave MoE layer forward.

TEST INFRASTRUCTURE ONLY: see the package docstring.  Nothing here is tuned;
each function does one step of the layer in the order the pages give it:

  router top-k  ->  latent down-projection  ->  fixed per-destination pools,
  3 same-shape waves, sender cap 1.10 and receiver cap 1.15, drops counted
  ->  SwiGLU experts on the received rows  ->  weighted combine  ->  up-
  projection plus the shared experts.

Readings where the pages are silent (each one is listed with its reason in
the design notes):

* gate weights: softmax over the k selected logits (the pages name no gate
  function);
* capacity: smallest integer >= cf x (uniform expected rows), the factor
  taken to six decimals, per wave slice for the sender cap, clamped to the
  most rows that can ever arrive;
* waves: wave w carries local experts [w*E_l/W, (w+1)*E_l/W) of every
  destination, so every (source, destination, wave) slice has one shape;
* drop priority: token index ascending, then top-k rank ascending; the
  receiver sees only sender-kept rows, in that order;
* a dropped assignment contributes zero (no renormalisation); the shared
  experts still see every token;
* combine in latent space, then one up-projection (linear-equivalent to
  projecting each expert output first).

Storage points that the layer keeps in bfloat16 (z, h, Y, c, the shared
activations, out) are rounded here with ``bf16_round``; everything else is
float64.  Router logits are rounded to float32, the precision in which the
top-k decision is taken.
"""
from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction
import math

import numpy as np

__all__ = [
    "bf16_round", "silu", "Plan", "make_plan", "router_logits", "router_topk",
    "latent_down", "placement", "dispatch", "pack_pool", "expert_ffn",
    "experts_forward", "combine", "shared_act", "output", "layer", "balance_update",
    "balance_update_window",
    "dispatch_ragged", "layer_ragged", "layer_backward", "silu_grad", "exact",
    "TIE_EPS", "EMPTY_TAG", "DROP_KEPT", "DROP_SEND", "DROP_RECV",
]

TIE_EPS = float(np.float32(1e-4))   # near-tie threshold on float32 logits
EMPTY_TAG = (-1, -1, -1, 0)          # tag of a pool slot nobody filled
DROP_KEPT, DROP_SEND, DROP_RECV = 0, 1, 2
CF_UNBOUNDED = 1e6                   # factors at or above this mean "no cap"


# ---------------------------------------------------------------- numerics

def bf16_round(a) -> np.ndarray:
    """Round to the nearest bfloat16 value, halves to even; float64 result.

    bfloat16 keeps 8 significant bits, so inside the binade [2^(e-1), 2^e)
    the representable values are the multiples of 2^(e-8); below 2^-126 the
    spacing stays 2^-133 (subnormals).  Magnitudes that round to 2^128 or
    more become infinities.
    """
    a = np.asarray(a, dtype=np.float64)
    out = a.copy()
    fin = np.isfinite(a)
    v = a[fin]
    _, e = np.frexp(v)
    e = np.maximum(e, -125)
    q = np.ldexp(1.0, e - 8)
    r = np.rint(v / q) * q                      # np.rint rounds halves to even
    big = np.abs(r) >= 2.0 ** 128
    r[big] = np.copysign(np.inf, v[big])
    out[fin] = r
    return out


def silu(g) -> np.ndarray:
    """SiLU (swish) in float64: g * sigmoid(g) = g / (1 + exp(-g))."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):                     # torch tensor (any dtype) -> float64
        a = a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- sizes

@dataclass(frozen=True)
class Plan:
    T: int
    S: int            # logical source ranks
    D: int            # logical destination ranks (= S)
    E: int
    k: int
    W: int            # waves
    T_s: int          # tokens per source
    E_l: int          # local experts per destination
    E_w: int          # local experts per wave
    c_send: int       # rows per (source, destination, wave) slice
    c_recv: int       # rows per expert
    pool_rows: int    # D * W * S * c_send


def _decimal(cf: float) -> Fraction:
    return Fraction(int(round(cf * 10 ** 6)), 10 ** 6)


def _capacity(cf: float, expected: Fraction, most: int) -> int:
    """Smallest integer >= cf * expected, clamped to the most rows possible."""
    if not math.isfinite(cf) or cf >= CF_UNBOUNDED:
        return most
    c = math.ceil(_decimal(cf) * expected)
    return max(0, min(c, most))


def make_plan(cfg) -> Plan:
    """Capacities and pool size.

    [LJ-HK] sec. 二: each source keeps one fixed pool per destination GPU; the
    sender capacity factor 1.10 bounds one source -> one destination, the
    receiver factor 1.15 bounds the rows of one local expert; the transfer is
    3 waves of identical shape.  Expected loads are the uniform ones:
    T_s*k/D rows per (source, destination), T*k/E rows per expert; the sender
    cap applies per wave slice of the pool.
    """
    T, E, k, W = cfg.T, cfg.n_experts, cfg.top_k, cfg.n_waves
    S = D = cfg.n_ranks
    if T % S or E % D or (E // D) % W or k > E or k < 1:
        raise ValueError("T must divide by the ranks, E by the ranks, E/ranks by the waves")
    T_s, E_l = T // S, E // D
    E_w = E_l // W
    c_send = _capacity(cfg.cf_send, Fraction(T_s * k, D * W), T_s * min(k, E_w))
    c_recv = _capacity(cfg.cf_recv, Fraction(T * k, E), T)
    return Plan(T, S, D, E, k, W, T_s, E_l, E_w, c_send, c_recv, D * W * S * c_send)


# ---------------------------------------------------------------- router

def router_logits(x, Wr, bias=None, dtype=np.float32) -> np.ndarray:
    """l = x Wr^T + bias, exact in float64, then rounded to float32 (``dtype``;
    float64 keeps it exact).

    [LJ-HK] sec. 二: the router picks experts per token; [CSDN] appendix A.2:
    the balancing bias is added to the router logits.
    """
    l = _f64(x) @ _f64(Wr).T
    if bias is not None:
        l = l + _f64(bias)[None, :]
    return l.astype(dtype)


def router_topk(l32, k: int, eps: float = TIE_EPS, dtype=np.float32):
    """Top-k experts per token, softmax gate weights and near-tie flags.

    [LJ-HK] sec. 二: the router selects eight experts for each token.
    Order: descending logit, equal logits -> lower expert id first.
    Weights: softmax over the k selected logits (reading; the pages name no
    gate function).  tie bit 0: the k-th and (k+1)-th logits differ by less
    than eps (the selected *set* is fragile); bit 1: two adjacent selected
    logits differ by less than eps (the *order*, hence the drop priority, is
    fragile).  Differences are exact (float64 of float32 values).
    """
    l = np.asarray(l32, dtype=dtype).astype(np.float64)
    T, E = l.shape
    order = np.argsort(-l, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    lsel = np.take_along_axis(l, order[:, :k], axis=1)
    ex = np.exp(lsel - lsel[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    tie = np.zeros(T, dtype=np.uint8)
    if k > 1:
        inner = (lsel[:, :-1] - lsel[:, 1:] < eps).any(axis=1)
        tie |= inner.astype(np.uint8) << 1
    if k < E:
        nxt = np.take_along_axis(l, order[:, k:k + 1], axis=1)[:, 0]
        tie |= (lsel[:, -1] - nxt < eps).astype(np.uint8)
    return idx, w, tie


# ---------------------------------------------------------------- latent

def latent_down(x, W_ld, rnd=bf16_round) -> np.ndarray:
    """z = bf16(x W_ld^T).  [LJ-HK] sec. 二: a latent projection compresses
    the routed activations from 6144 to 3072 values before the exchange."""
    return rnd(_f64(x) @ _f64(W_ld).T)


# ---------------------------------------------------------------- dispatch

def placement(e, p: Plan):
    """Destination rank, local id and wave of expert e (contiguous placement:
    E_l = E/D experts per destination, [LJ-HK] sec. 二 "six per GPU"; wave
    w carries local experts [w*E_w, (w+1)*E_w))."""
    e = np.asarray(e)
    dst = e // p.E_l
    q = e % p.E_l
    return dst, q, q // p.E_w


def _rank_within_key(keys: np.ndarray) -> np.ndarray:
    """For each position i: how many earlier positions hold the same key."""
    n = keys.shape[0]
    out = np.empty(n, dtype=np.int64)
    if n == 0:
        return out
    order = np.argsort(keys, kind="stable")
    sk = keys[order]
    starts = np.r_[0, np.nonzero(sk[1:] != sk[:-1])[0] + 1]
    lens = np.diff(np.r_[starts, n])
    first = np.repeat(starts, lens)
    out[order] = np.arange(n) - first
    return out


def dispatch(idx, p: Plan) -> dict:
    """Fixed pooled-wave dispatch with the two capacity caps.

    [LJ-HK] sec. 二: one fixed pool per destination, filled for 3 waves of one
    shape; the sender cap bounds one source -> one destination, the receiver
    cap bounds the rows of one local expert; any assignment that overflows
    either buffer is dropped and counted separately.

    Priority: assignments are visited in (token, top-k rank) order.  Sender
    stage: key (src, dst, wave); the n-th assignment with a key takes slot n
    if n < c_send, else it is dropped by the sender.  Receiver stage: the
    sender-kept assignments in the same order; the r-th one for expert e
    gets expert row r if r < c_recv, else it is dropped by the receiver (its
    pool slot stays filled but is never computed).
    Pool row of (dst, wave, src, slot) = ((dst*W + wave)*S + src)*c_send + slot.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    e = idx.reshape(-1)                                   # priority order
    tok = np.repeat(np.arange(T), k)
    src = tok // p.T_s if p.T_s else tok
    dst, _, wv = placement(e, p)
    key = (src * p.D + dst) * p.W + wv
    slot = _rank_within_key(key)
    send_kept = slot < p.c_send
    row = ((dst * p.W + wv) * p.S + src) * p.c_send + slot

    kept_pos = np.nonzero(send_kept)[0]
    r = _rank_within_key(e[kept_pos])
    recv_ok = r < p.c_recv

    drop = np.full(T * k, DROP_SEND, dtype=np.uint8)
    drop[kept_pos[recv_ok]] = DROP_KEPT
    drop[kept_pos[~recv_ok]] = DROP_RECV
    slot_of = np.full(T * k, -1, dtype=np.int32)
    slot_of[kept_pos[recv_ok]] = row[kept_pos[recv_ok]]
    send_row = np.where(send_kept, row, -1).astype(np.int64)

    expert_rows = np.full((p.E, p.c_recv), -1, dtype=np.int32)
    ok = kept_pos[recv_ok]
    expert_rows[e[ok], r[recv_ok]] = row[ok]
    count = np.bincount(e[ok], minlength=p.E).astype(np.int32)

    demand = np.bincount(key, minlength=p.S * p.D * p.W).reshape(p.S, p.D, p.W)
    recv_demand = np.bincount(e[kept_pos], minlength=p.E)
    stats = dict(
        assignments=T * k,
        kept=int(ok.size),
        dropped_send=int((~send_kept).sum()),
        dropped_recv=int((~recv_ok).sum()),
    )
    return dict(
        slot_of=slot_of.reshape(T, k), drop=drop.reshape(T, k), send_row=send_row.reshape(T, k),
        expert_rows=expert_rows, count=count, send_demand=demand,
        send_fill=np.minimum(demand, p.c_send), recv_demand=recv_demand, stats=stats,
    )


def pack_pool(z, idx, disp: dict, p: Plan, rows=None):
    """Payload rows and tags of the fixed pools.

    [LJ-HK] sec. 二: the expert id travels inside the activation payload, so
    no counts or routing metadata are exchanged separately.  A filled slot
    holds z[t] and the tag (expert, token, top-k rank, 0); an empty slot has
    tag (-1, -1, -1, 0) and no payload (NaN here).  ``rows`` restricts the
    result to a subset of pool rows (for large pools).
    """
    z = _f64(z)
    idx = np.asarray(idx)
    T, k = idx.shape
    rows = np.arange(p.pool_rows) if rows is None else np.asarray(rows)
    where = {}
    sr = disp["send_row"]
    for t, j in zip(*np.nonzero(sr >= 0)):
        where[int(sr[t, j])] = (int(t), int(j))
    payload = np.full((rows.size, z.shape[1]), np.nan)
    tags = np.tile(np.array(EMPTY_TAG, dtype=np.int32), (rows.size, 1))
    for i, r in enumerate(rows):
        tj = where.get(int(r))
        if tj is not None:
            t, j = tj
            payload[i] = z[t]
            tags[i] = (idx[t, j], t, j, 0)
    return payload, tags


# ---------------------------------------------------------------- experts

def expert_ffn(X, Wg_e, Wu_e, Wd_e, rnd=bf16_round) -> np.ndarray:
    """One routed expert on its rows: Y = bf16(bf16(silu(X Wg^T) * (X Wu^T)) Wd^T).

    [LJ-HK] sec. 二 / [CSDN] sec. 四: each receiver runs its local experts on
    the rows it received.  The pages name no activation; the layer sizes fix
    a SwiGLU expert (gate, up, down)."""
    X = _f64(X)
    g = X @ _f64(Wg_e).T
    u = X @ _f64(Wu_e).T
    h = rnd(silu(g) * u)
    return rnd(h @ _f64(Wd_e).T)


def experts_forward(payload_of_row, disp: dict, Wg, Wu, Wd, experts=None, rnd=bf16_round) -> dict:
    """Y for every computed pool row: {row: Y[row]} over experts' kept rows.

    ``payload_of_row(rows) -> X`` returns the pool payload of those rows."""
    out = {}
    E = disp["count"].shape[0]
    for e in (range(E) if experts is None else experts):
        n = int(disp["count"][e])
        if n == 0:
            continue
        rows = disp["expert_rows"][e, :n]
        Y = expert_ffn(payload_of_row(rows), Wg[e], Wu[e], Wd[e], rnd)
        for r, y in zip(rows, Y):
            out[int(r)] = y
    return out


# ---------------------------------------------------------------- combine

def combine(Y_of_row, slot_of, w, L: int, tokens=None, rnd=bf16_round) -> np.ndarray:
    """c[t] = bf16(sum over kept j, in j order, of w[t,j] * Y[slot_of[t,j]]).

    [LJ-HK] sec. 二: expert outputs come back to their tokens and are
    combined; a dropped assignment contributes nothing and the remaining
    weights are not renormalised (reading)."""
    slot_of = np.asarray(slot_of)
    w = _f64(w)
    T, k = slot_of.shape
    tokens = range(T) if tokens is None else tokens
    c = []
    for t in tokens:
        acc = np.zeros(L)
        for j in range(k):
            r = int(slot_of[t, j])
            if r >= 0:
                acc = acc + w[t, j] * _f64(Y_of_row(r))
        c.append(acc)
    return rnd(np.stack(c)) if c else np.zeros((0, L))


# ---------------------------------------------------------------- output

def shared_act(x, Wsg, Wsu, rnd=bf16_round) -> np.ndarray:
    """Shared-expert activations a_s = bf16(silu(x Wsg_s^T) * (x Wsu_s^T)),
    concatenated over s along the hidden axis.  [LJ-HK] sec. 二: two shared
    experts stay local and process every token."""
    x = _f64(x)
    Wsg, Wsu = _f64(Wsg), _f64(Wsu)
    parts = [rnd(silu(x @ Wsg[s].T) * (x @ Wsu[s].T)) for s in range(Wsg.shape[0])]
    return np.concatenate(parts, axis=1) if parts else np.zeros((x.shape[0], 0))


def output(c, a, W_lu, Wsd, rnd=bf16_round) -> np.ndarray:
    """out = bf16(c W_lu^T + sum_s a_s Wsd_s^T).

    [LJ-HK] sec. 二: the routed output is projected back to model width and
    then combined with the shared-expert path (unit weight)."""
    c, W_lu, Wsd = _f64(c), _f64(W_lu), _f64(Wsd)
    a = _f64(a)
    acc = c @ W_lu.T
    Hs = Wsd.shape[2] if Wsd.ndim == 3 else 0
    for s in range(Wsd.shape[0]):
        acc = acc + a[:, s * Hs:(s + 1) * Hs] @ Wsd[s].T
    return rnd(acc)


# ---------------------------------------------------------------- dropless ragged dispatch

def dispatch_ragged(idx, p: Plan) -> dict:
    """Dropless ragged dispatch, the pages' fallback if drops stay too high.

    [LJ-HK] sec. 四: a ragged all-to-all without drops.  Reading: the same
    destination-major pool order (destination, wave, source, priority), but
    each (source, destination, wave) block holds exactly the rows routed
    there, so blocks start at the exclusive prefix of the counts and the pool
    has T*k rows; nothing is dropped; expert e's rows, in priority order,
    are expert_rows[expert_offsets[e] : expert_offsets[e+1]].
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    e = idx.reshape(-1)
    tok = np.repeat(np.arange(T), k)
    src = tok // p.T_s if p.T_s else tok
    dst, _, wv = placement(e, p)
    gkey = (dst * p.W + wv) * p.S + src                  # block order in the pool
    slot = _rank_within_key(gkey)
    counts = np.bincount(gkey, minlength=p.D * p.W * p.S)
    block_start = np.r_[0, np.cumsum(counts)[:-1]]
    row = block_start[gkey] + slot
    r = _rank_within_key(e)
    ecount = np.bincount(e, minlength=p.E)
    eoff = np.r_[0, np.cumsum(ecount)]
    expert_rows = np.full(T * k, -1, dtype=np.int64)
    expert_rows[eoff[e] + r] = row
    return dict(slot_of=row.reshape(T, k).astype(np.int32), send_row=row.reshape(T, k),
                drop=np.zeros((T, k), dtype=np.uint8), expert_offsets=eoff.astype(np.int32),
                expert_rows=expert_rows.astype(np.int32), count=ecount.astype(np.int32),
                block_counts=counts.reshape(p.D, p.W, p.S),
                stats=dict(assignments=T * k, kept=T * k, dropped_send=0, dropped_recv=0))


def layer_ragged(cfg, t: dict) -> dict:
    """The whole layer with the dropless ragged dispatch."""
    p = make_plan(cfg)
    l32 = router_logits(t["x"], t["Wr"], t.get("bias"))
    idx, w, tie = router_topk(l32, cfg.top_k)
    z = latent_down(t["x"], t["W_ld"])
    disp = dispatch_ragged(idx, p)
    T, k = idx.shape
    payload = np.full((T * k, z.shape[1]), np.nan)
    tags = np.tile(np.array(EMPTY_TAG, dtype=np.int32), (T * k, 1))
    for tt in range(T):
        for j in range(k):
            rr = disp["slot_of"][tt, j]
            payload[rr] = z[tt]
            tags[rr] = (idx[tt, j], tt, j, 0)
    Y = {}
    for e in range(p.E):
        rows = disp["expert_rows"][disp["expert_offsets"][e]:disp["expert_offsets"][e + 1]]
        if rows.size:
            for rr, y in zip(rows, expert_ffn(payload[rows], t["Wg"][e], t["Wu"][e], t["Wd"][e])):
                Y[int(rr)] = y
    c = combine(lambda rr: Y[rr], disp["slot_of"], w, z.shape[1])
    a = shared_act(t["x"], t["Wsg"], t["Wsu"])
    out = output(c, a, t["W_lu"], t["Wsd"])
    return dict(plan=p, logits=l32, idx=idx, w=w, tie=tie, z=z, disp=disp, payload=payload,
                tags=tags, Y=Y, c=c, a=a, out=out)


# ---------------------------------------------------------------- backward pass

def silu_grad(g) -> np.ndarray:
    """d silu / dg = sigmoid(g) * (1 + g * (1 - sigmoid(g)))."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    return sig * (1.0 + g * (1.0 - sig))


def layer_backward(cfg, t: dict, fwd: dict, dout, rnd=bf16_round) -> dict:
    """Gradients of the layer output with respect to x and every weight.

    The pages give the forward only (the 250,691 tokens/s they report is a
    training step); this is its derivative, step by step in reverse:
      out = c W_lu^T + sum_s a_s Wsd_s^T      -> dc, da_s, dW_lu, dWsd_s
      a_s = silu(x Wsg_s^T) * (x Wsu_s^T)     -> dgs, dus, dWsg, dWsu
      c_t = sum_kept w_tj Y_row               -> dY_row = w_tj dc_t, dw_tj = <dc_t, Y_row>
      Y = h Wd^T, h = silu(g) u, g/u = X Wg^T / X Wu^T  (per expert)
                                              -> dh, dg, du, dX, dWd, dWg, dWu
      X_row = z_t (for every kept row)        -> dz_t = sum_kept dX_row
      z = x W_ld^T                            -> dW_ld
      w = softmax(l_selected), l = x Wr^T + b -> dl (zero off the selection), dWr
      x feeds z, l and the shared experts     -> dx
    The balancing bias gets no gradient (stop-gradient, [CSDN] appendix A.2).
    `rnd` is applied where the tensors are kept in bf16 (dc, da, dY, dh, dg,
    du, dX, dz, dl, dx); weight gradients stay float64.  Pre-activations g/u
    are recomputed in float64 from the stored inputs.
    """
    x = _f64(t["x"])
    W_lu, Wsd = _f64(t["W_lu"]), _f64(t["Wsd"])
    Wsg, Wsu = _f64(t["Wsg"]), _f64(t["Wsu"])
    dout = _f64(dout)
    p = fwd["plan"]
    T, k = fwd["idx"].shape
    L = W_lu.shape[1]
    ns, Hs = Wsd.shape[0], (Wsd.shape[2] if Wsd.ndim == 3 else 0)
    c, a = fwd["c"], fwd["a"]
    g_ = {}
    dc = rnd(dout @ W_lu)
    g_["W_lu"] = dout.T @ c
    dgs, dus = np.zeros((T, ns * Hs)), np.zeros((T, ns * Hs))
    g_["Wsd"] = np.zeros_like(Wsd)
    g_["Wsg"], g_["Wsu"] = np.zeros_like(Wsg), np.zeros_like(Wsu)
    for s_ in range(ns):
        sl = slice(s_ * Hs, (s_ + 1) * Hs)
        da = rnd(dout @ Wsd[s_])
        g_["Wsd"][s_] = dout.T @ a[:, sl]
        gs, us = x @ Wsg[s_].T, x @ Wsu[s_].T
        dgs[:, sl] = rnd(da * us * silu_grad(gs))
        dus[:, sl] = rnd(da * silu(gs))
        g_["Wsg"][s_] = dgs[:, sl].T @ x
        g_["Wsu"][s_] = dus[:, sl].T @ x
    # combine
    slot_of, w = fwd["disp"]["slot_of"], fwd["w"]
    dY, dw = {}, np.zeros((T, k))
    for tt in range(T):
        for j in range(k):
            r = int(slot_of[tt, j])
            if r >= 0:
                dY[r] = rnd(w[tt, j] * dc[tt])
                dw[tt, j] = dc[tt] @ fwd["Y"][r]
    # experts
    Wg, Wu, Wd = t["Wg"], t["Wu"], t["Wd"]
    g_["Wg"] = np.zeros(np.shape(Wg))
    g_["Wu"] = np.zeros(np.shape(Wu))
    g_["Wd"] = np.zeros(np.shape(Wd))
    dX = {}
    disp = fwd["disp"]
    lists = ([disp["expert_rows"][e, :disp["count"][e]] for e in range(p.E)]
             if "expert_offsets" not in disp else
             [disp["expert_rows"][disp["expert_offsets"][e]:disp["expert_offsets"][e + 1]]
              for e in range(p.E)])
    for e in range(p.E):
        rows = lists[e]
        if rows.size == 0:
            continue
        X = fwd["payload"][rows]
        Wg_e, Wu_e, Wd_e = _f64(Wg[e]), _f64(Wu[e]), _f64(Wd[e])
        gg, uu = X @ Wg_e.T, X @ Wu_e.T
        h = rnd(silu(gg) * uu)
        dYe = np.stack([dY[int(r)] for r in rows])
        dh = rnd(dYe @ Wd_e)
        g_["Wd"][e] = dYe.T @ h
        dg = rnd(dh * uu * silu_grad(gg))
        du = rnd(dh * silu(gg))
        g_["Wg"][e] = dg.T @ X
        g_["Wu"][e] = du.T @ X
        dXe = rnd(dg @ Wg_e + du @ Wu_e)
        for r, v in zip(rows, dXe):
            dX[int(r)] = v
    dz = np.zeros((T, L))
    for tt in range(T):
        for j in range(k):
            r = int(slot_of[tt, j])
            if r >= 0:
                dz[tt] += dX[r]
    dz = rnd(dz)
    g_["W_ld"] = dz.T @ x
    # router: softmax over the selected logits
    dl_sel = w * (dw - (w * dw).sum(axis=1, keepdims=True))
    dl = np.zeros((T, p.E))
    np.put_along_axis(dl, fwd["idx"].astype(np.int64), dl_sel, axis=1)
    dl = rnd(dl)
    g_["Wr"] = dl.T @ x
    dx = dz @ _f64(t["W_ld"]) + dl @ _f64(t["Wr"])
    for s_ in range(ns):
        sl = slice(s_ * Hs, (s_ + 1) * Hs)
        dx = dx + dgs[:, sl] @ Wsg[s_] + dus[:, sl] @ Wsu[s_]
    g_["x"] = rnd(dx)
    g_.update(dc=dc, dY=dY, dw=dw, dX=dX, dz=dz, dl=dl, dgs=dgs, dus=dus)
    return g_


# ---------------------------------------------------------------- balancing bias

def balance_update(idx, hist, alpha: float, n_experts: int):
    """Quantile-balancing bias for the next step.

    [CSDN] appendix A.2: a global histogram H counts how often each expert
    was selected; f_i = H[i] / sum(H); b_i = -alpha * (f_i - 1/E), added to
    the router logits from the next batch on (no gradient).  [CSDN] sec. 四
    describes the same update.  Reading: H counts top-k selections (before
    capacity drops), accumulated over the batches since the caller last
    cleared it (the caller's window); with an empty histogram b = 0.
    Returns (new histogram, bias) as (int64, float64) arrays.
    """
    idx = np.asarray(idx, dtype=np.int64).reshape(-1)
    h = np.asarray(hist, dtype=np.int64) + np.bincount(idx, minlength=n_experts)
    total = int(h.sum())
    if total == 0:
        return h, np.zeros(n_experts)
    f = h / total
    return h, -alpha * (f - 1.0 / n_experts)


def balance_update_window(idx, hist, ring, step: int, alpha: float, n_experts: int):
    """The same bias over the past N batches exactly ([CSDN] appendix A.2:
    H counts each expert's selections "in the past N batches").

    ring [N, E] holds batch b's counts in row b % N; this batch (number
    `step`, counted from 0) replaces the row of batch step - N, which leaves
    the window, so H = sum of the last N batches' counts.  [CSDN] sec. 四
    calls the histogram "10,000 bins"; read here as the window length N,
    the caller's choice.  Returns (hist, ring, step + 1, bias).
    """
    ring = np.array(ring, dtype=np.int64, copy=True)
    counts = np.bincount(np.asarray(idx, dtype=np.int64).reshape(-1), minlength=n_experts)
    slot = step % ring.shape[0]
    h = np.asarray(hist, dtype=np.int64) - ring[slot] + counts
    ring[slot] = counts
    total = int(h.sum())
    if total == 0:
        return h, ring, step + 1, np.zeros(n_experts)
    return h, ring, step + 1, -alpha * (h / total - 1.0 / n_experts)


# ---------------------------------------------------------------- layer

def exact(a) -> np.ndarray:
    """No rounding: the precision policy of a float64-throughout layer."""
    return np.asarray(a, dtype=np.float64)


def layer(cfg, t: dict, gate_w=None, rnd=bf16_round) -> dict:
    """The whole layer on one batch, every intermediate kept.

    ``t`` holds the inputs (x, Wr, bias, W_ld, Wg, Wu, Wd, W_lu, Wsg, Wsu,
    Wsd).  ``gate_w`` optionally overrides the gate weights (used by tests
    that zero the routed path).  ``rnd`` is the storage rounding (bf16 by
    default; ``exact`` gives a float64-throughout layer, logits included)."""
    p = make_plan(cfg)
    ldt = np.float64 if rnd is exact else np.float32
    l32 = router_logits(t["x"], t["Wr"], t.get("bias"), dtype=ldt)
    idx, w, tie = router_topk(l32, cfg.top_k, dtype=ldt)
    if gate_w is not None:
        w = np.asarray(gate_w, dtype=np.float64)
    z = latent_down(t["x"], t["W_ld"], rnd)
    disp = dispatch(idx, p)
    payload, tags = pack_pool(z, idx, disp, p)
    # expert weights are widened to float64 one expert at a time (inside expert_ffn)
    Y = experts_forward(lambda rows: payload[np.asarray(rows)], disp, t["Wg"], t["Wu"], t["Wd"],
                        rnd=rnd)
    L = z.shape[1]
    c = combine(lambda r: Y[r], disp["slot_of"], w, L, rnd=rnd)
    a = shared_act(t["x"], t["Wsg"], t["Wsu"], rnd)
    out = output(c, a, t["W_lu"], t["Wsd"], rnd)
    return dict(plan=p, logits=l32, idx=idx, w=w, tie=tie, z=z, disp=disp,
                payload=payload, tags=tags, Y=Y, c=c, a=a, out=out)
