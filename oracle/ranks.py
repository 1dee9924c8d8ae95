"""Oracle for the multi-device planner (test infrastructure; see the package
docstring).

"Window-Aligned Sequence Parallelism (SeedVR2)":

* §Planner -- a deterministic LPT assignment: windows sorted by
  (-video token count, original window id); each window goes to the rank
  with the smallest (assigned tokens, rank id); each rank then lists its
  windows in ascending original order.
* §Plan A redistribution -- with Z_src[r] / Z_dst[d] the canonical token ids
  held by each rank and C[r, d] the number of rows rank d needs from rank r:
  rank r's input split sizes are row r of C and its output split sizes are
  column r; each peer segment is packed in destination-local order, so the
  receiver reorders with one argsort of the concatenated destination
  positions; the exchange is needed iff some row changes rank (computed from
  the global C, so every rank takes the same branch).

Written with Python lists and sets, one rule at a time, in the order above.
"""
import numpy as np


def lpt_assign(sizes, world):
    """Window -> rank by the §Planner rules; returns (win_rank, rank_tokens)."""
    order = sorted(range(len(sizes)), key=lambda w: (-int(sizes[w]), w))
    load = [0] * world
    win_rank = [0] * len(sizes)
    for w in order:
        r = min(range(world), key=lambda rr: (load[rr], rr))
        win_rank[w] = r
        load[r] += int(sizes[w])
    return win_rank, load


def rank_tokens(win_off, ids, win_rank, rank):
    """Canonical ids held by `rank`, in its local order (windows ascending)."""
    out = []
    for w in range(len(win_off) - 1):
        if win_rank[w] == rank:
            out.extend(int(c) for c in ids[win_off[w]:win_off[w + 1]])
    return out


def exchange(src, dst, world):
    """Plan A tables.  src / dst = (win_off, ids) of the two layouts.
    Returns (C, exchange_required, send_rows[r], recv_pos[d])."""
    ws, _ = lpt_assign(np.diff(src[0]), world)
    wd, _ = lpt_assign(np.diff(dst[0]), world)
    Zs = [rank_tokens(*src, ws, r) for r in range(world)]
    Zd = [rank_tokens(*dst, wd, d) for d in range(world)]
    C = np.array([[len(set(Zs[r]) & set(Zd[d])) for d in range(world)] for r in range(world)],
                 dtype=np.int64)
    required = any(C[r, d] for r in range(world) for d in range(world) if r != d)
    send, recv = [], []
    for r in range(world):
        src_local = {c: i for i, c in enumerate(Zs[r])}
        rows = []
        for d in range(world):  # segment for d, in d's local order
            rows.extend(src_local[c] for c in Zd[d] if c in src_local)
        send.append(rows)
    for d in range(world):
        dst_local = {c: i for i, c in enumerate(Zd[d])}
        pos = []
        for r in range(world):  # segments arrive in source-rank order
            held = set(Zs[r])
            pos.extend(dst_local[c] for c in Zd[d] if c in held)
        recv.append(pos)
    return C, required, send, recv
