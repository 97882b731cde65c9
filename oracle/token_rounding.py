"""Token rounding (TR) routing and the dropless layer on variable expert sets:
CPU oracle, written from the pages. TEST INFRASTRUCTURE ONLY: the product path
never imports this module.

Source: "SonicMoE" notes, 3.4.4 "Token Rounding Routing" (Algorithm 4 with the
NR-f round-and-sparsify subroutine):
  1. token-choice top-K on the router scores; f_e = tokens that chose expert e;
  2. the two tile multiples floor(f_e) and ceil(f_e) (to M_tile);
  3. a biased score S' = S for the token-choice pairs and S - 1 for the others,
     so that token-choice tokens always rank first;
  4. per expert, tokens sorted by S' (descending); keep ceil(f_e) tokens (pad
     with the best expert-choice tokens) if ceil(f_e) - f_e < f_e - floor(f_e),
     else floor(f_e) tokens (drop the lowest-scoring token-choice tokens).

Readings where the pages are silent (each is stated where it is used):
  * S is the softmax of the router logits over all experts (the router's
    probabilities); equal S' rank the lower token id first.
  * A tie in NR-f (equal distance to both multiples) and an exact multiple
    both keep floor(f_e) = f_e tokens when f_e is a multiple; a tie rounds down.
  * An expert cannot keep more tokens than exist: n_e = min(n_e, T).
  * The gate weights of a token are the softmax of its logits over its final
    expert set (renormalised over the chosen experts, as for top-K routing); a
    token left without experts contributes nothing and gets no gradient.
  * An expert's final rows are in ascending token order; a token's experts in
    ascending expert id, which is also the order its outputs are summed in.

Everything is float64 on the given values.
"""
from __future__ import annotations

import numpy as np

from oracle.moe_oracle import _as64, act, act_grad, silu, silu_grad, softmax


def token_rounding(z, K: int, m_tile: int = 128, ids=None):
    """Token rounding of the logits z [T, E]. Returns a dict:
    final [T,E] bool (the rounded assignment), w [T,E] (gate weights, zero off
    the final set), tc [T,E] bool (the token-choice assignment), f [E]
    (token-choice counts), n [E] (kept counts), up [E] bool (padded), p [T,E]
    (the scores). `ids` [T,K] gives the token-choice assignment instead of
    taking the top-K of z (to compare on another implementation's routing)."""
    z = _as64(z)
    T, E = z.shape
    p = softmax(z)
    if ids is None:
        ids = np.argsort(-p, axis=1, kind="stable")[:, :K]   # token choice, ties to lower id
    ids = np.asarray(ids, dtype=np.int64)
    tc = np.zeros((T, E), dtype=bool)
    tc[np.arange(T)[:, None], ids] = True
    f = tc.sum(axis=0).astype(np.int64)
    lo = (f // m_tile) * m_tile
    hi = -((-f) // m_tile) * m_tile
    up = (hi - f) < (f - lo)
    n = np.minimum(np.where(up, hi, lo), T)
    final = np.zeros((T, E), dtype=bool)
    tok = np.arange(T)
    for e in range(E):
        s_biased = np.where(tc[:, e], p[:, e], p[:, e] - 1.0)
        order = np.lexsort((tok, -s_biased))              # S' descending, then token ascending
        final[order[: n[e]], e] = True
    w = np.zeros((T, E))
    for t in range(T):
        sel = final[t]
        if sel.any():
            w[t, sel] = softmax(z[t, sel])
    return dict(final=final, w=w, tc=tc, f=f, n=n, up=up, p=p)


def rows_of(final):
    """The rounded assignment as rows: expert_token_indices [N] (each expert's
    tokens ascending), offsets [E+1], and per token the rows of its experts in
    ascending expert order: tok_off [T+1], tok_exp [N], tok_rows [N]."""
    final = np.asarray(final, dtype=bool)
    T, E = final.shape
    counts = final.sum(axis=0)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    eti = np.concatenate([np.nonzero(final[:, e])[0] for e in range(E)]).astype(np.int64) \
        if offsets[E] else np.zeros(0, dtype=np.int64)
    row = -np.ones((T, E), dtype=np.int64)
    for e in range(E):
        row[eti[offsets[e]:offsets[e + 1]], e] = np.arange(offsets[e], offsets[e + 1])
    n_t = final.sum(axis=1)
    tok_off = np.zeros(T + 1, dtype=np.int64)
    tok_off[1:] = np.cumsum(n_t)
    tok_exp = np.concatenate([np.nonzero(final[t])[0] for t in range(T)]).astype(np.int64) \
        if tok_off[T] else np.zeros(0, dtype=np.int64)
    tok_rows = np.array([row[t, e] for t in range(T) for e in np.nonzero(final[t])[0]],
                        dtype=np.int64)
    return dict(eti=eti, offsets=offsets, tok_off=tok_off, tok_exp=tok_exp, tok_rows=tok_rows)


def _ffn(xe, W1e, W3e, W2e, expert):
    a = xe @ W1e.T
    if expert == "swiglu":
        b = xe @ W3e.T
        A = silu(a) * b
    else:
        b = None
        A = act(a, expert)
    return a, b, A, A @ W2e.T


def layer_forward_sets(x, W1, W3, W2, final, w, expert: str = "swiglu"):
    """Dropless forward on variable expert sets: y_t = sum over e in final(t),
    ascending e, of w[t,e] * E_e(x_t). Returns y [T,d] and per-expert (a, b, A, Y)
    in each expert's ascending token order."""
    x = _as64(x)
    W1, W2 = _as64(W1), _as64(W2)
    W3 = _as64(W3) if expert == "swiglu" else None
    final = np.asarray(final, dtype=bool)
    w = _as64(w)
    T, E = final.shape
    y = np.zeros((T, x.shape[1]))
    per = []
    for e in range(E):
        toks = np.nonzero(final[:, e])[0]
        a, b, A, Y = _ffn(x[toks], W1[e], None if W3 is None else W3[e], W2[e], expert)
        per.append((toks, a, b, A, Y))
    for t in range(T):                      # slot order = ascending expert id
        for e in np.nonzero(final[t])[0]:
            toks, _, _, _, Y = per[e]
            y[t] += w[t, e] * Y[np.searchsorted(toks, t)]
    return dict(y=y, per=per)


def layer_backward_sets(dO, x, Wg, W1, W3, W2, final, w, fwd=None, expert: str = "swiglu"):
    """Gradients of L = <dO, y> for the set-based layer: dx, dWg, dW1, dW3
    (None when non-gated), dW2 and dS [T,E] = <dO_t, Y_{t,e}> on the final set.
    The router gradient differentiates w[t, .] = softmax of z_t over final(t):
    dz_e = w_e (dS_e - sum_j w_j dS_j) on final(t), zero elsewhere."""
    dO = _as64(dO)
    x = _as64(x)
    Wg, W1, W2 = _as64(Wg), _as64(W1), _as64(W2)
    gated = expert == "swiglu"
    W3 = _as64(W3) if gated else None
    final = np.asarray(final, dtype=bool)
    w = _as64(w)
    if fwd is None:
        fwd = layer_forward_sets(x, W1, W3, W2, final, w, expert)
    T, E = final.shape
    dx = np.zeros_like(x)
    dW1 = np.zeros_like(W1)
    dW3 = np.zeros_like(W3) if gated else None
    dW2 = np.zeros_like(W2)
    dS = np.zeros((T, E))
    for e in range(E):
        toks, a, b, A, Y = fwd["per"][e]
        if len(toks) == 0:
            continue
        we = w[toks, e][:, None]
        dS[toks, e] = np.sum(dO[toks] * Y, axis=1)
        dY = we * dO[toks]
        dW2[e] = dY.T @ A
        dA = dY @ W2[e]
        if gated:
            da = dA * b * silu_grad(a)
            db = dA * silu(a)
            dW3[e] = db.T @ x[toks]
            dx[toks] += db @ W3[e]
        else:
            da = dA * act_grad(a, expert)
        dW1[e] = da.T @ x[toks]
        dx[toks] += da @ W1[e]
    sbar = np.sum(w * dS, axis=1, keepdims=True)
    dz = np.where(final, w * (dS - sbar), 0.0)
    dWg = dz.T @ x
    dx += dz @ Wg
    return dict(dx=dx, dWg=dWg, dW1=dW1, dW3=dW3, dW2=dW2, dS=dS, dz=dz)
