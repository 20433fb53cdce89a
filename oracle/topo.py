"""Two-domain collective scheduler of HOCCL section 3.4 (oracle).

Topology: G GPUs in nodes (NVLink domains); every GPU u has a symmetric peer
sym[u] in the same node (the GPU under the same PCIe switch, the one that
holds u's RDMA staging buffers).  One RDMA domain connects the nodes.

Traffic matrix abstraction (Eqs. 2-5).  The origin matrix C[u][v] holds the
logical flow from u to v.  An inter-node flow m = C[u][v] is carried as a
sender-side NVLink forwarding copy f'_m on (u, sym[u]), the RDMA transfer f_m
(accounted at cell (u, v)), and a receiver-side forwarding copy f''_m on
(sym[v], v).  With A_u = sum of u's outgoing inter-node flows and B_v = sum of
v's incoming inter-node flows,

    T[u][v] = C[u][v] + A_u + B_v   if (u, v) is intra-node and v = sym[u]
    T[u][v] = C[u][v]               otherwise.

Stage decomposition (Algorithm 1, Eqs. 6-11), taken step by step:
  1. residual R <- T, P <- empty;
  2. decompose the native intra-node traffic (C's intra-node entries) of each
     NVLink domain into matching components;
  3. while inter-node traffic remains:
  4.   new stage T^s;
  5.   extract a contention-free RDMA matching (at most one outgoing and one
       incoming inter-node flow per GPU, Eq. 8);
  6.   move the largest removable portion of it -- the smallest residual among
       the matched flows -- into T^s;
  7.   add the matching sender-side and receiver-side forwarding copies;
  8.   fill the NVLink slack with native matching components;
  9.   append T^s to P.
Stage time tau^s = max over domains of L^s_d / B_d with L^s_d the largest
entry of domain d in T^s (Eqs. 9-10); the objective is sum tau^s (Eq. 11).

Readings where the pages leave a step open (also listed in the design notes):
  * matchings (steps 2 and 5) are built greedily: candidate entries sorted by
    size descending, then by (u, v); an entry is taken if its row and column
    are still free;
  * step 8's slack: a stage of duration tau^s lets every NVLink cell carry up
    to tau^s * B_nvlink bytes; native components are added in the order step 2
    produced them, each by the largest amount that keeps every cell of its
    matching within that capacity (integer bytes, floor);
  * native traffic left after the inter-node traffic is exhausted: the NVLink
    domains run in parallel, so each further stage takes the next remaining
    matching of every domain (duration = the largest of them / B_nvlink);
  * bandwidths are integers (bytes per unit time) so capacities are exact:
    when the RDMA term binds, cap = floor(x * B_nv / B_rdma); otherwise the
    stage is NVLink-bound and cap is its largest NVLink entry.
"""
from __future__ import annotations


def domains(node_of):
    G = len(node_of)
    inter = {(u, v) for u in range(G) for v in range(G) if u != v and node_of[u] != node_of[v]}
    intra = {(u, v) for u in range(G) for v in range(G) if u != v and node_of[u] == node_of[v]}
    return inter, intra


def traffic_matrix(C, node_of, sym):
    """HOCCL traffic matrix T (Eq. 4) from the origin matrix C."""
    G = len(C)
    inter, _ = domains(node_of)
    A = [sum(C[u][v] for v in range(G) if (u, v) in inter) for u in range(G)]
    B = [sum(C[u][v] for u in range(G) if (u, v) in inter) for v in range(G)]
    T = [[C[u][v] for v in range(G)] for u in range(G)]
    for u in range(G):
        v = sym[u]
        if v != u and node_of[v] == node_of[u]:
            T[u][v] += A[u] + B[v]
    return T


def greedy_matching(entries):
    """entries: {(u, v): size > 0}.  Largest first, ties by (u, v); one per row and column."""
    rows, cols, picked = set(), set(), []
    for (u, v), size in sorted(entries.items(), key=lambda e: (-e[1], e[0][0], e[0][1])):
        if u in rows or v in cols:
            continue
        rows.add(u)
        cols.add(v)
        picked.append((u, v))
    return picked


def native_components(C, node_of):
    """Step 2: per NVLink domain, peel matchings off the native intra-node traffic."""
    G = len(C)
    comps = []
    for d in sorted(set(node_of)):
        N = {(u, v): C[u][v] for u in range(G) for v in range(G)
             if u != v and node_of[u] == d and node_of[v] == d and C[u][v] > 0}
        while N:
            M = greedy_matching(N)
            w = min(N[e] for e in M)
            comps.append([M, w])
            for e in M:
                N[e] -= w
                if N[e] == 0:
                    del N[e]
    return comps


def schedule(C, node_of, sym, bw_nvlink: int, bw_rdma: int):
    """Returns (T, stages, taus): stages are G x G integer matrices, taus their durations."""
    G = len(C)
    inter, intra = domains(node_of)
    T = traffic_matrix(C, node_of, sym)
    R = {(u, v): C[u][v] for (u, v) in inter if C[u][v] > 0}
    comps = native_components(C, node_of)
    stages, taus = [], []
    while R:
        S = [[0] * G for _ in range(G)]
        M = greedy_matching(R)
        x = min(R[e] for e in M)
        for (u, v) in M:
            S[u][v] += x
            R[(u, v)] -= x
            if R[(u, v)] == 0:
                del R[(u, v)]
            S[u][sym[u]] += x          # sender-side forwarding copy f'
            S[sym[v]][v] += x          # receiver-side forwarding copy f''
        l_nv = max([S[u][v] for (u, v) in intra] or [0])
        if x * bw_nvlink >= l_nv * bw_rdma:      # RDMA-bound stage
            cap = (x * bw_nvlink) // bw_rdma
            tau = x / bw_rdma
        else:                                     # NVLink-bound stage
            cap = l_nv
            tau = l_nv / bw_nvlink
        for comp in comps:
            Mn, w = comp
            if w == 0:
                continue
            room = min(cap - S[u][v] for (u, v) in Mn)
            a = min(w, room)
            if a > 0:
                for (u, v) in Mn:
                    S[u][v] += a
                comp[1] = w - a
        stages.append(S)
        taus.append(tau)
    # Leftover native traffic: the NVLink domains run in parallel, so every
    # further stage takes the next remaining matching of each domain.
    queues = {}
    for Mn, w in comps:
        if w > 0:
            queues.setdefault(node_of[Mn[0][0]], []).append((Mn, w))
    while any(queues.values()):
        S = [[0] * G for _ in range(G)]
        longest = 0
        for d in sorted(queues):
            if not queues[d]:
                continue
            Mn, w = queues[d].pop(0)
            for (u, v) in Mn:
                S[u][v] = w
            longest = max(longest, w)
        stages.append(S)
        taus.append(longest / bw_nvlink)
    return T, stages, taus
