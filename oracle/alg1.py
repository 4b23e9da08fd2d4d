"""The pull-based dispatch schedule of "Mixture-of-Kittens: MoE Megakernel
for NVL72s", Sec. 3.1 (Algorithm 1), for any number of ranks R -- TEST
INFRASTRUCTURE (pure Python, for small inputs).

Inputs: routes A[r][j] in {0..R*L-1} (expert of route j on source rank r),
the receiving rank c and L local experts per rank.  Output: Phi, where
Phi[P] = (r, j) says that buffer position P of rank c receives route j of
rank r.  Sec. 3.1 states what the table is: each local expert gets one
contiguous region, the regions in expert order, and inside a region the
routes arrive round-robin over the source ranks -- every rank's first route
to that expert, then every rank's second one, and so on, ranks ascending
within a round.

Two independent statements of that one permutation (the tests compare them):
``alg1_schedule`` counts and scans -- M[r][l] routes from rank r to local
expert l, region starts S by an exclusive prefix sum of the per-expert totals
-- and then fills each region by merging the per-rank route queues
round-robin; ``sort_key_schedule`` sorts the routes by the key (local expert,
ordinal o of the route among its rank's routes to that expert, source rank r).
"""
from __future__ import annotations


def alg1_schedule(A, c: int, L: int):
    R = len(A)
    lo = c * L
    # per (local expert, source rank): that rank's routes to the expert, in route order
    queues = [[[] for _ in range(R)] for _ in range(L)]
    for r in range(R):
        for j, a in enumerate(A[r]):
            if lo <= a < lo + L:
                queues[a - lo][r].append(j)
    M = [[len(queues[l][r]) for l in range(L)] for r in range(R)]
    # regions in expert order: exclusive prefix sum of the per-expert totals
    S = []
    start = 0
    for l in range(L):
        S.append(start)
        start += sum(M[r][l] for r in range(R))
    Phi = []
    for l in range(L):
        depth = max((M[r][l] for r in range(R)), default=0)
        for rnd in range(depth):  # round rnd: every rank's (rnd+1)-th route to expert l
            for r in range(R):
                if rnd < M[r][l]:
                    Phi.append((r, queues[l][r][rnd]))
        assert len(Phi) == S[l] + sum(M[r][l] for r in range(R))
    return Phi, M, S


def sort_key_schedule(A, c: int, L: int):
    keys = []
    for r in range(len(A)):
        for j, a in enumerate(A[r]):
            if c * L <= a < (c + 1) * L:
                o = sum(1 for jp in range(j) if A[r][jp] == a)
                keys.append(((a - c * L, o, r), (r, j)))
    keys.sort(key=lambda kv: kv[0])
    return [rj for _, rj in keys]
