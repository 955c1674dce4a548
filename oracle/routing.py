"""Route validity, expert_map remap, capacity and route packing.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix (flashinfer PR #4255):

* Description: "Shape-stable route packing: the triton packing kernels
  specialize on a power-of-two capacity instead of the exact token count ...
  The W4A16 workspaces are sized to the same capacity."
* Tests: route packing is checked "against a host reference, covering
  expert_map, invalid expert ids, preallocated buffers, and the workspace
  capacity contract".
* Review comments: ``route_pack_token_capacity(topk)`` takes a top-k it does
  not use, and the packed-route and route-block capacities are clamped to at
  least 1.

Readings taken:

* capacity: T_cap = next_pow2(max(m, 1)) tokens, R_cap = T_cap * top_k routes;
* a route (t, j) with id = ids[t, j] is valid iff 0 <= id < E_g and
  l = expert_map[id] (or id when there is no map) satisfies 0 <= l < E_l;
  invalid routes are dropped, never an error;
* routes are flattened as r = t * top_k + j; inside each expert's list they
  keep ascending r (a stable counting sort), which makes packing bit-exact;
* entries of sorted_routes past the number of valid routes hold -1.
"""

from __future__ import annotations

import numpy as np


def next_pow2(n: int) -> int:
    n = int(n)
    p = 1
    while p < n:
        p *= 2
    return p


def route_capacity_tokens(m: int) -> int:
    """Token capacity the packing and workspaces are sized to: next_pow2(max(m, 1))."""
    return next_pow2(max(int(m), 1))


def route_capacity(m: int, top_k: int) -> int:
    """Route capacity R_cap = T_cap * top_k, clamped to at least 1."""
    return max(route_capacity_tokens(m) * int(top_k), 1)


def local_experts(ids, num_global_experts, num_local_experts, expert_map=None):
    """Local expert of every route, or -1 for a dropped route.  ids: [m, k]."""
    ids = np.asarray(ids, dtype=np.int64)
    valid = (ids >= 0) & (ids < num_global_experts)
    safe = np.where(valid, ids, 0)
    if expert_map is None:
        loc = safe
    else:
        em = np.asarray(expert_map, dtype=np.int64)
        if em.shape != (num_global_experts,):
            raise ValueError("expert_map must have one entry per global expert")
        loc = em[safe]
    valid &= (loc >= 0) & (loc < num_local_experts)
    return np.where(valid, loc, -1)


def route_pack(ids, num_global_experts, num_local_experts, expert_map=None):
    """Pack valid routes by local expert.

    Returns (counts [E_l] int32, offsets [E_l + 1] int32,
    sorted_routes [R_cap] int32).  offsets is the exclusive scan of counts
    with offsets[E_l] = number of valid routes; sorted_routes[offsets[l] + i]
    is the i-th valid route of expert l in ascending flat index; the tail is -1.
    """
    ids = np.asarray(ids, dtype=np.int64)
    m, k = ids.shape
    loc = local_experts(ids, num_global_experts, num_local_experts, expert_map).reshape(-1)
    counts = np.zeros(num_local_experts, dtype=np.int64)
    for l in loc:
        if l >= 0:
            counts[l] += 1
    offsets = np.zeros(num_local_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    cap = route_capacity(m, k)
    sorted_routes = np.full(cap, -1, dtype=np.int64)
    fill = offsets[:-1].copy()
    for r, l in enumerate(loc):  # ascending flat route index -> stable
        if l >= 0:
            sorted_routes[fill[l]] = r
            fill[l] += 1
    return counts.astype(np.int32), offsets.astype(np.int32), sorted_routes.astype(np.int32)
