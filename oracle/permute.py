"""S4: token-to-expert permutation (oracle; test infrastructure only).

Pairs are the (token, slot) picks of the router, numbered p = t * k + j.  The
permutation groups them by expert: a histogram of the picks per expert, its
exclusive prefix sum and a stable scatter, so that inside one expert the pairs
keep token order.  The pages do not describe this step; it is the plainest
form of the grouping that a grouped expert GEMM needs.

  counts[e]  number of pairs routed to expert e
  offsets    exclusive prefix sum of counts, length E + 1 (offsets[E] = number
             of computed pairs: T * k, fewer when a route-tail skip dropped some)
  perm[r]    pair id at position r of the expert-grouped order
  inv[p]     position of pair p in that order (inv[perm[r]] = r); -1 for a
             pair the route-tail skip dropped (expert index -1)
"""
import numpy as np


def permute(idx, num_experts: int):
    idx = np.asarray(idx, dtype=np.int64)
    pair_expert = idx.reshape(-1)
    pairs = pair_expert.size
    live = np.nonzero(pair_expert >= 0)[0]            # pairs that are computed
    counts = np.bincount(pair_expert[live], minlength=num_experts).astype(np.int32)
    offsets = np.zeros(num_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = live[np.argsort(pair_expert[live], kind="stable")].astype(np.int32)
    inv = np.full(pairs, -1, dtype=np.int32)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offsets, perm, inv
