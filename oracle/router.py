"""S1/S2: router logits, top-k and renormalised softmax weights (oracle;
test infrastructure only).

Reading taken (the pages only say that every expert the router picks is
computed -- capy-flash status post, "Where it stands"):
  * logits l[t, e] = sum_h x[t, h] * Wr[e, h] (+ b[e]) on the unquantised bf16
    activations, evaluated here in float64;
  * the k experts with the largest logits are picked, ordered by (logit
    descending, expert index ascending), so exact ties go to the lower index;
  * weights w_j = exp(l_j - l_0) / sum_{j' < k} exp(l_j' - l_0) over the picks
    only (the same as a full softmax restricted to the picks and renormalised).

Route-tail skip (optional).  The capy-flash status post ("Where it stands")
credits another engine's faster single-card decode mostly to a "route tail
skip" that drops low-ranked experts which miss its expert cache, while
capy-flash computes every pick.  Reading taken: with a keep count r
(1 <= r <= k), the picks at ranks 0 .. r-1 are always computed; a pick at rank
j >= r is computed only if its expert is marked resident (the cache of the
pages; with no residency mask nothing is resident, so the whole tail is
dropped).  The weights are renormalised over the kept picks only,
w_j = exp(l_j - l_0) / sum_{kept j'} exp(l_j' - l_0).  A dropped pick keeps
its slot with expert index -1 and weight 0.  r = k (or no skip) is the layer
above.
"""
import numpy as np


def router_logits(x, router_w, bias=None) -> np.ndarray:
    """float64 logits [T][E] from x [T][H] and Wr [E][H] (+ bias [E])."""
    logits = np.asarray(x, dtype=np.float64) @ np.asarray(router_w, dtype=np.float64).T
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=np.float64)[None, :]
    return logits


def topk_full_sort(logits, k: int) -> np.ndarray:
    """Indices [T][k] of the top-k logits per row by a full sort on
    (-logit, expert index)."""
    logits = np.asarray(logits, dtype=np.float64)
    rows, experts = logits.shape
    expert_ids = np.broadcast_to(np.arange(experts), (rows, experts))
    # np.lexsort sorts by the last key first: primary -logit, then expert index
    order = np.lexsort((expert_ids, -logits), axis=-1)
    return order[:, :k].astype(np.int32)


def renormalised_softmax(selected_logits) -> np.ndarray:
    """Softmax over the k selected logits of each row (slot 0 is the largest)."""
    sel = np.asarray(selected_logits, dtype=np.float64)
    z = np.exp(sel - sel[:, :1])
    return z / np.sum(z, axis=1, keepdims=True)


def kept_picks(idx, keep, resident=None) -> np.ndarray:
    """Boolean [T][k]: which picks the route-tail skip computes (rank < keep,
    or an expert marked resident)."""
    idx = np.asarray(idx)
    rank = np.broadcast_to(np.arange(idx.shape[1]), idx.shape)
    kept = rank < keep
    if resident is not None:
        kept = kept | (np.asarray(resident)[idx] != 0)
    return kept


def route(logits, k: int, keep=None, resident=None):
    """Top-k indices [T][k] (int32) and their weights [T][k] (float64).

    keep: None (compute every pick) or the route-tail skip's keep count r;
    resident: None or a per-expert mask [E] of experts that are never skipped.
    Skipped picks get index -1 and weight 0; the weights of the kept picks are
    renormalised over the kept picks."""
    idx = topk_full_sort(logits, k)
    sel = np.take_along_axis(np.asarray(logits, dtype=np.float64), idx.astype(np.int64), axis=1)
    if keep is None or keep >= k:
        return idx, renormalised_softmax(sel)
    kept = kept_picks(idx, keep, resident)
    z = np.where(kept, np.exp(sel - sel[:, :1]), 0.0)
    w = z / np.sum(z, axis=1, keepdims=True)
    return np.where(kept, idx, -1).astype(np.int32), w


def near_tie_tokens(logits, k: int, tau: float) -> np.ndarray:
    """Boolean [T]: tokens whose ordered top-(k+1) logits have an adjacent gap
    below tau.  For those tokens an fp32 evaluation of the logits may order or
    pick the experts differently, so parity checks treat them separately."""
    logits = np.asarray(logits, dtype=np.float64)
    kk = min(k + 1, logits.shape[1])
    idx = topk_full_sort(logits, kk)
    sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    if kk < 2:
        return np.zeros(logits.shape[0], dtype=bool)
    gaps = sel[:, :-1] - sel[:, 1:]
    return np.any(gaps < tau, axis=1)
