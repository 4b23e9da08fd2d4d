"""Algorithm 1 ("Pull-based dispatch schedule construction") of
"Mixture-of-Kittens: MoE Megakernel for NVL72s", Sec. 3.1, for any number of
ranks R -- TEST INFRASTRUCTURE (pure Python, for small inputs).

Inputs: routes A[r][j] in {0..R*L-1} (expert of route j on source rank r),
the current rank c and L local experts per rank.  Output: Phi, where
Phi[P] = (r, j) says that local buffer position P receives route j of rank r.

``alg1_schedule`` evaluates the algorithm's closed form for the position p;
``sort_key_schedule`` is the same table read as Sec. 3.1 describes it: the
routes sorted by (local expert, per-source-rank ordinal o, source rank r).
The two are independent statements of one permutation; the tests compare them.
"""
from __future__ import annotations


def alg1_schedule(A, c: int, L: int):
    R = len(A)
    # route count per (source rank, local expert)
    M = [[0] * L for _ in range(R)]
    for r in range(R):
        for a in A[r]:
            if c * L <= a < (c + 1) * L:
                M[r][a - c * L] += 1
    # start of each local expert's region
    S = [0] * L
    for l in range(1, L):
        S[l] = S[l - 1] + sum(M[r][l - 1] for r in range(R))
    total = S[L - 1] + sum(M[r][L - 1] for r in range(R)) if L else 0
    Phi = [None] * total
    for r in range(R):
        for j, a in enumerate(A[r]):
            if not (c * L <= a < (c + 1) * L):
                continue
            l = a - c * L
            # o: earlier routes of this source rank to the same expert
            o = sum(1 for jp in range(j) if A[r][jp] == a)
            p = sum(min(M[rp][l], o) for rp in range(R)) + sum(1 for rp in range(r) if M[rp][l] > o)
            Phi[S[l] + p] = (r, j)
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
