"""Brute-force layouts for tiny inputs, by a definition independent of moe_ref.c.

TEST INFRASTRUCTURE ONLY.  Where the oracle builds its layouts by counting and
exclusive scans (the pages' method: "Enabling trillion-parameter models on AWS
EFA", sections "Send and receive buffers" and "Dispatch and combine"), this
module lists every (token, expert) assignment and sorts the list with Python's
``sorted`` on explicit keys.  Both must give the same positions.

  send row of (s, t, k) in sender s's buffer:   rank order of key (p(e), e, t, k)
      among s's assignments -- contiguous per peer, then per expert;
  grouped row in receiver r's layout:           rank order of key (e, s, t, k)
      among the assignments whose expert lives on r -- per local expert, then
      per sender (the grouped-GEMM layout);
  combine send row in expert rank r's buffer:   rank order of key (s, e, t, k)
      among the same assignments -- contiguous per destination s, and in s's
      own send order within it.

Expert e lives on rank p(e) = e // (E // N).  Ids outside [0, E) take no row.
"""
from __future__ import annotations

import itertools

import numpy as np


def assignments(N: int, T: int, E: int, R: int, idx: np.ndarray):
    idx = np.asarray(idx).reshape(N, T, R)
    return [(s, t, k, int(idx[s, t, k])) for s in range(N) for t in range(T) for k in range(R)
            if 0 <= int(idx[s, t, k]) < E]


def layouts(N: int, T: int, E: int, R: int, idx: np.ndarray):
    """Return (send_row, grp_row, csend_row): dicts keyed by (s, t, k)."""
    Er = E // N
    asg = assignments(N, T, E, R, idx)
    send_row, grp_row, csend_row = {}, {}, {}
    for s in range(N):
        mine = sorted((a for a in asg if a[0] == s), key=lambda a: (a[3] // Er, a[3], a[1], a[2]))
        for pos, a in enumerate(mine):
            send_row[a[:3]] = pos
    for r in range(N):
        here = [a for a in asg if a[3] // Er == r]
        for pos, a in enumerate(sorted(here, key=lambda a: (a[3], a[0], a[1], a[2]))):
            grp_row[a[:3]] = pos
        for pos, a in enumerate(sorted(here, key=lambda a: (a[0], a[3], a[1], a[2]))):
            csend_row[a[:3]] = pos
    return send_row, grp_row, csend_row


def all_routings(N: int, T: int, E: int, R: int):
    """Every routing in which each token picks R distinct experts, in order."""
    per_token = list(itertools.permutations(range(E), R))
    for combo in itertools.product(per_token, repeat=N * T):
        yield np.array(combo, dtype=np.int32).reshape(N, T, R)


def ll_rows(N: int, T: int, E: int, R: int, idx: np.ndarray) -> dict:
    """Low-latency row of every (s, t, k): region (receiver r, local expert j,
    sender s) of T rows, position = rank of (t, k) in sorted order among
    sender s's assignments to that expert; None beyond T rows."""
    Er = E // N
    rows = {}
    for s in range(N):
        for e in range(E):
            mine = sorted(a for a in assignments(N, T, E, R, idx) if a[0] == s and a[3] == e)
            r, j = e // Er, e % Er
            for u, a in enumerate(mine):
                rows[a[:3]] = ((r * Er + j) * N + s) * T + u if u < T else None
    return rows
