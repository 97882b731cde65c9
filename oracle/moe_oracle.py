"""CPU oracle of the dropless token-choice MoE layer (forward and backward).

TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the bench's
CPU-baseline leg may import this module. The product path never calls it, and
it shares no code with the CUDA library: it is a plain, slow, fp64 statement of
what the layer computes, so that the GPU kernels can be checked against it.

Sources (page title, section):
  [MB-notes]  MoEBlaze: Breaking the Memory Wall for Efficient MoE Training on
              Modern GPUs (paper notes): 2.1 gating, 2.3 aggregation, 4.1 data
              structures and Fig. 2, 5.1 SwiGLU, 5.2 Algorithm 1.
  [MB-expl]   MoEBlaze explainer: 3.4 "Dispatch Data Structures", "Fused
              SwiGLU Kernel with Activation Checkpoint".
  [Sonic]     SonicMoE: Accelerating MoE with IO and Tile-aware Optimizations,
              3.4.1 memory-efficient backward pass.
  [Dropless]  Dropless MoE, in depth: "The dropless forward pass, step by
              step", "A reference implementation", "Worked example: one
              skewed batch".

Readings where the pages are silent or disagree (each one is a choice):
  * The router renormalises over the chosen K experts ([Dropless] reference
    implementation); the MoEBlaze gating formula has no renormalisation.
  * Top-K ties go to the lower expert id; slot 0 holds the largest weight.
  * A router bias, when given, is added to the logits before the softmax.
  * SiLU goes on the gate projection W1; W3 is the up projection and W2 the
    down projection (MoEBlaze's Algorithm 1 names them W1, W2, W3 = gate, up,
    down; SonicMoE fuses gate/up into one W1).
  * Within one expert, tokens are in ascending token order (stable sort).
  * The K expert outputs of a token are summed in slot order k = 0..K-1.
  * The renormalised weights equal a softmax over the K chosen logits (the
    full-softmax denominator cancels), so the router backward is the Jacobian
    of that K-way softmax, with zero gradient for unchosen experts.
  * Non-gated experts ([MB-notes] 2.2, E_i(x) = W_2,i s(W_1,i x), with the
    SiLU or ReLU activation of the MoEBlaze configurations): a = W1 x,
    A = act(a), Y = W2 A; W3 is absent and the saved pre-activation is a.

Everything is computed in float64 on the given values (the callers round
activations and weights to bf16 first).
"""
from __future__ import annotations

import numpy as np

f64 = np.float64


def _as64(a) -> np.ndarray:
    """Any array-like (numpy or torch CPU tensor) as a float64 numpy array."""
    if hasattr(a, "detach"):
        a = a.detach().float().numpy() if a.dtype.is_floating_point else a.detach().numpy()
    return np.asarray(a, dtype=f64)


def _asint(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().numpy()
    return np.asarray(a, dtype=np.int64)


# --------------------------------------------------------------------------
# Router: logits, softmax, top-K, renormalisation
# [MB-notes] 2.1 (TopK(softmax(W_g x)), W_g in R^{E x d});
# [Dropless] "A reference implementation" (softmax, topk, renormalise over k).
# --------------------------------------------------------------------------
def softmax(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def route(x, Wg, K: int, bias=None):
    """Returns (z [T,E], p [T,E], ids [T,K] int64, w [T,K]).

    z = x W_g^T (+ bias); p = softmax(z); ids = the K largest p in descending
    order, ties to the lower expert id; w = p[ids] / sum p[ids]."""
    x = _as64(x)
    Wg = _as64(Wg)
    z = x @ Wg.T
    if bias is not None:
        z = z + _as64(bias)[None, :]
    p = softmax(z)
    # A stable sort of -p keeps equal probabilities in ascending expert order.
    ids = np.argsort(-p, axis=1, kind="stable")[:, :K]
    pk = np.take_along_axis(p, ids, axis=1)
    w = pk / pk.sum(axis=1, keepdims=True)
    return z, p, ids, w


def topk_gap(z: np.ndarray, K: int) -> np.ndarray:
    """Per token, the smallest logit gap that decides the top-K set or its
    order: min over consecutive sorted logits among the first K+1."""
    zs = -np.sort(-z, axis=1)
    m = min(K + 1, z.shape[1])
    if m < 2:
        return np.full(z.shape[0], np.inf)
    return np.min(zs[:, : m - 1] - zs[:, 1:m], axis=1)


# --------------------------------------------------------------------------
# Dispatch index
# [MB-notes] 4.1 (expert_token_indices, expert_token_offsets,
# token_expert_indices, token_index_map; worked example of Fig. 2);
# [Dropless] "step by step" (stable sort by expert id, bincount).
# --------------------------------------------------------------------------
def build_dispatch(ids, E: int):
    """Returns (expert_token_indices [TK], expert_token_offsets [E+1],
    token_index_map [TK], counts [E]); all int64.

    The (token, slot) assignments, flattened token-major, are stably sorted by
    expert id; the sorted order lists each expert's tokens in ascending token
    order. token_index_map[t*K + k] is the position of assignment (t, k) in
    that sorted list."""
    ids = _asint(ids)
    T, K = ids.shape
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    eti = order // K
    counts = np.bincount(flat, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    tim = np.empty(T * K, dtype=np.int64)
    tim[order] = np.arange(T * K, dtype=np.int64)
    return eti, offsets, tim, counts


def tile_rows(counts, block: int = 128):
    """Per-expert M-tile counts and rows after rounding each expert's row count
    up to a multiple of `block` ([Dropless] "Worked example: one skewed batch")."""
    counts = _asint(counts)
    tiles = (counts + block - 1) // block
    return tiles, tiles * block


# --------------------------------------------------------------------------
# Expert FFN (SwiGLU) and the weighted combine
# [MB-notes] 5.1 (a = x W1, b = x W2, SiLU(a) * b); 2.2 (E_i(x) = W_2,i s(W_1,i x));
# [Sonic] 3.4.1 (H = X W1, A = SwiGLU(H), Y = A W2, O_t = sum_e pi s Y).
# --------------------------------------------------------------------------
def sigmoid(u: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-u))


def silu(u: np.ndarray) -> np.ndarray:
    return u * sigmoid(u)


def silu_grad(u: np.ndarray) -> np.ndarray:
    """d SiLU / du = s + u s (1 - s), s = sigmoid(u) ([MB-expl], fused SwiGLU)."""
    s = sigmoid(u)
    return s + u * s * (1.0 - s)


EXPERTS = ("swiglu", "silu", "relu")


def relu(u: np.ndarray) -> np.ndarray:
    return np.maximum(u, 0.0)


def relu_grad(u: np.ndarray) -> np.ndarray:
    return (u > 0).astype(np.float64)


def act(u: np.ndarray, expert: str) -> np.ndarray:
    """Activation of a non-gated expert."""
    return silu(u) if expert == "silu" else relu(u)


def act_grad(u: np.ndarray, expert: str) -> np.ndarray:
    return silu_grad(u) if expert == "silu" else relu_grad(u)


def expert_ffn(xe: np.ndarray, W1e: np.ndarray, W3e, W2e: np.ndarray, expert: str = "swiglu"):
    """One expert on its rows. SwiGLU: a = xe W1e^T, b = xe W3e^T,
    A = SiLU(a) * b, Y = A W2e^T. Non-gated: a = xe W1e^T, A = act(a),
    Y = A W2e^T (b is None). W1e, W3e are [h, d]; W2e is [d, h] (out x in)."""
    a = xe @ W1e.T
    if expert == "swiglu":
        b = xe @ W3e.T
        A = silu(a) * b
    else:
        b = None
        A = act(a, expert)
    Y = A @ W2e.T
    return a, b, A, Y


def _w3(W3, expert):
    return _as64(W3) if expert == "swiglu" else None


def layer_forward(x, W1, W3, W2, ids, w, expert: str = "swiglu"):
    """Dropless forward with given routing. Returns dict with
    y [T,d], H (saved pre-activations per sorted row: [TK, 2h] = (a | b) for
    SwiGLU, [TK, h] = a otherwise), A [TK,h], Y [TK,d] (sorted row order) and
    the dispatch index."""
    x = _as64(x)
    W1, W3, W2 = _as64(W1), _w3(W3, expert), _as64(W2)
    ids = _asint(ids)
    w = _as64(w)
    T, K = ids.shape
    E, h, d = W1.shape
    gated = expert == "swiglu"
    eti, offsets, tim, counts = build_dispatch(ids, E)
    H = np.zeros((T * K, 2 * h if gated else h))
    A = np.zeros((T * K, h))
    Y = np.zeros((T * K, d))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        xe = x[eti[lo:hi]]                       # read rows in place, no routed copy kept
        a, b, Ae, Ye = expert_ffn(xe, W1[e], W3[e] if gated else None, W2[e], expert)
        H[lo:hi, :h] = a
        if gated:
            H[lo:hi, h:] = b
        A[lo:hi] = Ae
        Y[lo:hi] = Ye
    # [MB-notes] 2.3: y = sum over chosen experts of g_i(x) E_i(x), slot order.
    y = np.zeros((T, d))
    for k in range(K):
        rows = tim.reshape(T, K)[:, k]
        y += w[:, k:k + 1] * Y[rows]
    return dict(y=y, H=H, A=A, Y=Y, eti=eti, offsets=offsets, tim=tim, counts=counts)


def dense_forward(x, W1, W3, W2, ids, w, expert: str = "swiglu"):
    """Every expert on every token, then masked by the routing weights (a
    dense restatement used to pin the sparse forward on small inputs)."""
    x = _as64(x)
    W1, W3, W2 = _as64(W1), _w3(W3, expert), _as64(W2)
    ids = _asint(ids)
    w = _as64(w)
    T, K = ids.shape
    E = W1.shape[0]
    gate = np.zeros((T, E))
    for k in range(K):
        gate[np.arange(T), ids[:, k]] += w[:, k]
    y = np.zeros((T, x.shape[1]))
    for e in range(E):
        _, _, _, Ye = expert_ffn(x, W1[e], None if W3 is None else W3[e], W2[e], expert)
        y += gate[:, e:e + 1] * Ye
    return y


# --------------------------------------------------------------------------
# Backward
# [MB-notes] 3.2 and Algorithm 1 (FusedBackward); [MB-expl] backward via
# reverse indexing; [Sonic] 3.4.1 (dS_{t,e} = <dO_t, Y_{e,t}>).
# --------------------------------------------------------------------------
def router_backward_dz(w: np.ndarray, dS: np.ndarray) -> np.ndarray:
    """Gradient w.r.t. the K chosen logits of each token.

    w = softmax over the chosen logits, so dz = J^T dS with the K x K Jacobian
    J = diag(w) - w w^T. Unchosen logits get zero gradient."""
    T, K = w.shape
    dz = np.zeros((T, K))
    for t in range(T):
        J = np.diag(w[t]) - np.outer(w[t], w[t])
        dz[t] = J.T @ dS[t]
    return dz


def layer_backward(dO, x, Wg, W1, W3, W2, ids, w, fwd=None, expert: str = "swiglu"):
    """Hand-written backward with given routing. Returns dict with
    dx [T,d], dWg [E,d], dW1, dW3 [E,h,d] (dW3 None for non-gated experts),
    dW2 [E,d,h], dS [T,K], dz [T,K]."""
    dO = _as64(dO)
    x = _as64(x)
    Wg = _as64(Wg)
    W1, W3, W2 = _as64(W1), _w3(W3, expert), _as64(W2)
    ids = _asint(ids)
    w = _as64(w)
    T, K = ids.shape
    E, h, d = W1.shape
    gated = expert == "swiglu"
    if fwd is None:
        fwd = layer_forward(x, W1, W3, W2, ids, w, expert)
    eti, offsets, tim = fwd["eti"], fwd["offsets"], fwd["tim"]
    H, Y = fwd["H"], fwd["Y"]
    timm = tim.reshape(T, K)

    # Router-score gradient, plain definition: dS_{t,k} = <dO_t, Y_{t,k}>.
    dS = np.zeros((T, K))
    for k in range(K):
        dS[:, k] = np.sum(dO * Y[timm[:, k]], axis=1)

    # Per-row weight and upstream gradient of each expert output row:
    # dY_r = w_{t,k} dO_t (the combine's backward, scattered to routed rows).
    wrow = np.zeros(T * K)
    wrow[timm.reshape(-1)] = w.reshape(-1)
    dW1 = np.zeros_like(W1)
    dW3 = np.zeros_like(W3) if gated else None
    dW2 = np.zeros_like(W2)
    dxr = np.zeros((T * K, d))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        toks = eti[lo:hi]
        xe = x[toks]
        dY = wrow[lo:hi, None] * dO[toks]
        a = H[lo:hi, :h]
        dA = dY @ W2[e]                     # Y = A W2e^T  =>  dA = dY W2e
        if gated:
            b = H[lo:hi, h:]
            A = silu(a) * b
            da = dA * b * silu_grad(a)
            db = dA * silu(a)
            dW3[e] = db.T @ xe
            dxr[lo:hi] = da @ W1[e] + db @ W3[e]
        else:
            A = act(a, expert)
            da = dA * act_grad(a, expert)
            dxr[lo:hi] = da @ W1[e]
        dW2[e] = dY.T @ A
        dW1[e] = da.T @ xe
    # Token-gradient accumulation over the K routed rows, slot order.
    dx = np.zeros((T, d))
    for k in range(K):
        dx += dxr[timm[:, k]]

    # Router: dz over chosen logits, scattered into a dense [T,E] gradient.
    dzk = router_backward_dz(w, dS)
    dz = np.zeros((T, E))
    for k in range(K):
        dz[np.arange(T), ids[:, k]] += dzk[:, k]
    dWg = dz.T @ x
    dx = dx + dz @ Wg
    return dict(dx=dx, dWg=dWg, dW1=dW1, dW3=dW3, dW2=dW2, dS=dS, dz=dzk)


def layer_step(x, Wg, W1, W3, W2, dO, K: int, bias=None, expert: str = "swiglu"):
    """Route, dispatch, forward and backward of one layer step (all fp64)."""
    z, p, ids, w = route(x, Wg, K, bias)
    fwd = layer_forward(x, W1, W3, W2, ids, w, expert)
    bwd = layer_backward(dO, x, Wg, W1, W3, W2, ids, w, fwd, expert)
    return dict(z=z, p=p, ids=ids, w=w, fwd=fwd, bwd=bwd)


# --------------------------------------------------------------------------
# The same definitions evaluated on a sample (for parity at full size, where
# the whole layer is too slow on the CPU). Each is the plain definition above,
# restricted to the requested tokens or hidden units.
# --------------------------------------------------------------------------
def tokens_forward_backward(tokens, x, dO, Wg, W1, W3, W2, ids, w, expert: str = "swiglu"):
    """For the given tokens: y_t, dS_t, the expert part of dx_t, and dx_t with
    the router term. Works one token at a time with matrix-vector products."""
    tokens = _asint(tokens)
    ids = _asint(ids)
    w = _as64(w)
    K = ids.shape[1]
    d = W1.shape[2]
    Wg = _as64(Wg)
    out_y = np.zeros((len(tokens), d))
    out_dS = np.zeros((len(tokens), K))
    out_dx = np.zeros((len(tokens), d))
    cache = {}

    gated = expert == "swiglu"

    def weights(e):
        if e not in cache:
            cache[e] = (_as64(W1[e]), _as64(W3[e]) if gated else None, _as64(W2[e]))
        return cache[e]

    for i, t in enumerate(tokens):
        xt = _as64(x[t])
        dOt = _as64(dO[t])
        Ys = []
        dx_e = np.zeros(d)
        for k in range(K):
            e = int(ids[t, k])
            W1e, W3e, W2e = weights(e)
            a = W1e @ xt
            if gated:
                b = W3e @ xt
                A = silu(a) * b
            else:
                A = act(a, expert)
            Yk = W2e @ A
            Ys.append(Yk)
            out_y[i] += w[t, k] * Yk
            dA = W2e.T @ (w[t, k] * dOt)
            if gated:
                da = dA * b * silu_grad(a)
                db = dA * silu(a)
                dx_e += W1e.T @ da + W3e.T @ db
            else:
                da = dA * act_grad(a, expert)
                dx_e += W1e.T @ da
        dS = np.array([dOt @ Yk for Yk in Ys])
        out_dS[i] = dS
        dzk = router_backward_dz(w[t:t + 1], dS[None, :])[0]
        dx_r = np.zeros(d)
        for k in range(K):
            dx_r += dzk[k] * Wg[int(ids[t, k])]
        out_dx[i] = dx_e + dx_r
    return out_y, out_dS, out_dx


def hidden_unit_grads(e: int, j: int, x, dO, W1, W3, W2, ids, w, expert: str = "swiglu"):
    """For expert e and hidden unit j: dW1[e][j,:], dW3[e][j,:] (None for
    non-gated experts) and dW2[e][:,j], each summed over the tokens routed to e."""
    ids = _asint(ids)
    w = _as64(w)
    T, K = ids.shape
    sel_t, sel_k = np.nonzero(ids == e)
    d = W1.shape[2]
    gated = expert == "swiglu"
    if len(sel_t) == 0:
        return np.zeros(d), (np.zeros(d) if gated else None), np.zeros(d)
    xe = _as64(x[sel_t])
    dY = w[sel_t, sel_k][:, None] * _as64(dO[sel_t])
    W2e_j = _as64(W2[e][:, j])
    a = xe @ _as64(W1[e][j])
    dA = dY @ W2e_j
    if gated:
        b = xe @ _as64(W3[e][j])
        A = silu(a) * b
        da = dA * b * silu_grad(a)
        db = dA * silu(a)
        return da @ xe, db @ xe, dY.T @ A
    A = act(a, expert)
    da = dA * act_grad(a, expert)
    return da @ xe, None, dY.T @ A


def tokens_forward_backward_batched(tokens, x, dO, Wg, W1, W3, W2, ids, w,
                                    expert: str = "swiglu"):
    """Same outputs as tokens_forward_backward (y_t, dS_t and dx_t with the
    router term, for the given distinct tokens), evaluated one expert at a time
    over the sampled (token, slot) pairs routed to it, with matrix products.
    The expert FFN and its backward are the definitions of layer_forward and
    layer_backward ([MB-notes] 5.1, Algorithm 1; [Sonic] 3.4.1), restricted to
    the sampled tokens; a token's K expert outputs are added in fp64."""
    tokens = _asint(tokens)
    ids = _asint(ids)
    w = _as64(w)
    d = W1.shape[2]
    K = ids.shape[1]
    gated = expert == "swiglu"
    sub_ids = ids[tokens]
    sub_w = w[tokens]
    n = len(tokens)
    y = np.zeros((n, d))
    dS = np.zeros((n, K))
    dx = np.zeros((n, d))
    for e in np.unique(sub_ids):
        ii, kk = np.nonzero(sub_ids == e)      # a token meets expert e at most once
        xe = _as64(x[tokens[ii]])
        dOe = _as64(dO[tokens[ii]])
        W1e = _as64(W1[e])
        W2e = _as64(W2[e])
        a = xe @ W1e.T
        if gated:
            W3e = _as64(W3[e])
            b = xe @ W3e.T
            A = silu(a) * b
        else:
            A = act(a, expert)
        Y = A @ W2e.T
        wk = sub_w[ii, kk][:, None]
        y[ii] += wk * Y
        dS[ii, kk] = np.sum(dOe * Y, axis=1)
        dA = (wk * dOe) @ W2e
        if gated:
            da = dA * b * silu_grad(a)
            db = dA * silu(a)
            dx[ii] += da @ W1e + db @ W3e
        else:
            da = dA * act_grad(a, expert)
            dx[ii] += da @ W1e
    dz = router_backward_dz(sub_w, dS)
    Wg = _as64(Wg)
    for k in range(K):
        dx += dz[:, k:k + 1] * Wg[sub_ids[:, k]]
    return y, dS, dx


def hidden_units_grads(e: int, js, x, dO, W1, W3, W2, ids, w, expert: str = "swiglu"):
    """hidden_unit_grads for several hidden units js of expert e at once:
    dW1[e][js, :], dW3[e][js, :] (None for non-gated experts) and dW2[e][:, js],
    each summed over the tokens routed to e."""
    ids = _asint(ids)
    w = _as64(w)
    js = _asint(js)
    sel_t, sel_k = np.nonzero(ids == e)
    d = W1.shape[2]
    gated = expert == "swiglu"
    if len(sel_t) == 0:
        z = np.zeros((len(js), d))
        return z, (z.copy() if gated else None), np.zeros((d, len(js)))
    xe = _as64(x[sel_t])
    dY = w[sel_t, sel_k][:, None] * _as64(dO[sel_t])
    a = xe @ _as64(W1[e][js]).T
    dA = dY @ _as64(W2[e][:, js])
    if gated:
        b = xe @ _as64(W3[e][js]).T
        A = silu(a) * b
        da = dA * b * silu_grad(a)
        db = dA * silu(a)
        return da.T @ xe, db.T @ xe, dY.T @ A
    A = act(a, expert)
    da = dA * act_grad(a, expert)
    return da.T @ xe, None, dY.T @ A
