"""CPU model of the persistent attention kernel's barrier protocol.

The kernel (csrc/attn_tc.cu) coordinates a TMA producer, an MMA-issuing
warp, two softmax warpgroups (and, in the RoPE kernels, two warps that
rotate each item's Q tiles between the TMA landing and the MMA)
through mbarriers that are waited on by phase parity; work items reach all
roles through a ring of four slots filled from a global counter.  This model replays each role's sequence of waits, arrivals
and commits (a commit arrives when the MMAs before it finish; here, at once)
in random interleavings over real work-item lists, and checks that:
  * no interleaving deadlocks, and
  * every parity wait passes only at the phase it means: try_wait.parity(m&1)
    also passes when the barrier is one phase *behind* the target, or two
    ahead, so either would be a silent protocol error on the GPU.
A second simulation runs several CTAs at once, their producers drawing
items from one global counter in the kernel's order, so that each CTA's
item list is whatever the interleaving gives it (as on the GPU), also when
one CTA falls behind.
The sequences mirror attn_tc_kernel's roles; a change to the kernel's
protocol must be made here too and checked before it runs on a GPU.
"""
import random

import numpy as np
import pytest

from oracle import plan as op

def all_items(grid, L, heads, layout=op.REGULAR):
    """Every work item in the kernel's order (head h, then window w, then the
    (w, h) pairs of query tiles) as (w, h, nkv, nq, t0, vt)."""
    BM=128
    off, _ = op.layout_tables(*grid, layout)
    sizes=np.diff(off); nwin=len(sizes)
    tt=(L+BM-1)//BM
    out=[]
    for h in range(heads):
        for w in range(nwin):
            vt=int((sizes[w]+BM-1)//BM); nkv=vt+tt
            for jp in range((nkv+1)//2):
                out.append((w, h, nkv, min(2, nkv-2*jp), 2*jp, vt))
    return out


def items_for(grid, L, heads, nblocks, b, layout=op.REGULAR):
    """Work items that persistent CTA b walks when the items are dealt round
    robin (one of the orders the global counter can produce)."""
    return all_items(grid, L, heads, layout)[b::nblocks]


class Static:
    """A fixed item list: consumer u gets items[u], then the end mark."""
    def __init__(self, items):
        self.items = items

    def draw(self, u):
        return self.items[u] if u < len(self.items) else None

    get = draw


NRING = 4


def counts(rope):
    """Arrivals that complete one phase of each barrier (the model's roles
    stand for whole warps or warpgroups, one arrival each)."""
    c = {b: 1 for b in ('q_full', 'q_empty', 'pl_full0', 'pl_full1', 'pl_empty0', 'pl_empty1',
                        's_full0', 's_full1', 'p_full0', 'p_full1', 'o_full0', 'o_full1',
                        'o_empty0', 'o_empty1', 'q_ready')}
    for u in range(NRING):
        c['item_full%d' % u] = 1
        c['item_empty%d' % u] = 4 if rope else 3    # MMA, two softmax warpgroups (+ RoPE warps)
    return c


def take(u):
    """A consumer's share of the item ring for its u-th item (or the end mark)."""
    yield ('wait', 'item_full%d' % (u % NRING), u // NRING)
    yield ('arrive', 'item_empty%d' % (u % NRING))


def producer(src):
    # Items come from a global counter; the producer publishes each index in
    # ring slot u % 4 once the consumers have all read the index four back.
    # payload e (global): item start -> [K(g0)]; step j -> [V(g0+j), K(g0+j+1)] (K only if
    # the item has tile j+1).  Payload e lives in slot e&1; it may load once payload e-2
    # is released (its tiles use the same K/V stages).
    e=0; k=0
    for u in range(1 << 30):
        if u >= NRING: yield ('wait', 'item_empty%d' % (u % NRING), u // NRING - 1)
        item = src.draw(u)
        yield ('arrive', 'item_full%d' % (u % NRING))
        if item is None: break
        (w, h, nkv, nq, t0, vt) = item
        if k>0: yield ('wait','q_empty',k-1)
        yield ('arrive','q_full'); k+=1
        for p in range(nkv+1):
            if e>=2: yield ('wait','pl_empty%d'%(e&1),(e>>1)-1)
            yield ('arrive','pl_full%d'%(e&1))
            e+=1

def mma(src, rope):
    e=0; k=0; cs=[0,0]; co=[0,0]
    for u in range(1 << 30):
        yield from take(u)
        item = src.get(u)
        if item is None: break
        (w, h, nkv, nq, t0, vt) = item
        yield ('wait','q_ready' if rope else 'q_full',k)     # RoPE kernels: Q rotated
        yield ('wait','pl_full%d'%(e&1),e>>1)                # payload [K(0)]
        for i in range(nq): yield ('commit','s_full%d'%i)
        if nkv==1: yield ('commit','q_empty')
        yield ('commit','pl_empty%d'%(e&1))            # K(0) read by the S(0) just issued
        e+=1
        for j in range(nkv):
            more=j+1<nkv
            yield ('wait','pl_full%d'%(e&1),e>>1)      # payload [V(j), K(j+1)]
            for i in range(nq):
                yield ('wait','p_full%d'%i,cs[i]+j)
                if j==0 and co[i]>0: yield ('wait','o_empty%d'%i,co[i]-1)
                yield ('commit',('s_full%d' if more else 'o_full%d')%i)
            yield ('commit','pl_empty%d'%(e&1))        # V(j) and K(j+1) read by MMAs just issued
            if j+2==nkv: yield ('commit','q_empty')
            e+=1
        for i in range(nq): cs[i]+=nkv; co[i]+=1
        k+=1

def softmax(src,i):
    cs=0; co=0
    for u in range(1 << 30):
        yield from take(u)
        item = src.get(u)
        if item is None: break
        (w, h, nkv, nq, t0, vt) = item
        if i>=nq: continue
        for j in range(nkv):
            yield ('wait','s_full%d'%i,cs+j)
            yield ('arrive','p_full%d'%i)
        cs+=nkv
        yield ('wait','o_full%d'%i,co)
        yield ('arrive','o_empty%d'%i); co+=1

def rope_warps(src):
    # RoPE kernels: rotate the item's Q tiles between the TMA landing and the
    # MMA (K arrives rotated; K/V payloads go from the TMA to the MMA).
    k=0
    for u in range(1 << 30):
        yield from take(u)
        item = src.get(u)
        if item is None: break
        yield ('wait','q_full',k); yield ('arrive','q_ready'); k+=1

def simulate(items, seed, rope=False, lag=None):
    """Random interleaving; a role index in `lag` is picked only when nothing
    else is ready or with probability 1/20, so that it falls behind."""
    rnd=random.Random(seed)
    need=counts(rope)
    done={b:0 for b in need}      # completed phases
    arr={b:0 for b in need}       # arrivals in the current phase
    src=Static(items)
    roles=[producer(src),mma(src, rope),softmax(src,0),softmax(src,1)]
    if rope: roles.append(rope_warps(src))
    pending=[next(r,None) for r in roles]
    steps=0
    while any(p is not None for p in pending):
        ready=[]
        for idx,op_ in enumerate(pending):
            if op_ is None: continue
            if op_[0]=='wait':
                b,m=op_[1],op_[2]
                # hardware: try_wait.parity(m&1) passes iff (completed phases & 1) != (m & 1)
                if (done[b] & 1) != (m & 1):
                    assert done[b] == m + 1, ("parity wait passes at the wrong phase", op_, done[b], idx)
                    ready.append(idx)
            else: ready.append(idx)
        if not ready:
            raise RuntimeError("DEADLOCK: %s" % pending)
        if lag is not None and len(ready) > 1 and lag in ready and rnd.random() >= 0.05:
            ready.remove(lag)
        idx=rnd.choice(ready)
        op_=pending[idx]
        if op_[0] in ('arrive','commit'):
            b = op_[1]
            arr[b] += 1
            if arr[b] == need[b]:
                arr[b] = 0
                done[b] += 1
        pending[idx]=next(roles[idx],None); steps+=1
    return steps

CASES = [((2, 45, 80, 1, 3, 3), 16, 2, 152), ((2, 45, 80, 1, 3, 3), 16, 2, 7), ((3, 30, 40, 2, 3, 3), 300, 2, 5),
         ((3, 30, 40, 2, 3, 3), 0, 2, 3), ((21, 68, 120, 4, 3, 3), 256, 1, 40), ((2, 45, 80, 1, 9, 16), 3, 2, 11),
         ((2, 3, 200, 1, 1, 9), 0, 1, 2)]


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("layout", [op.REGULAR, op.SHIFTED])
@pytest.mark.parametrize("grid,L,heads,nb", CASES)
def test_protocol_has_no_deadlock_and_exact_parity(grid, L, heads, nb, layout, rope):
    for b in range(min(nb, 4)):
        its = items_for(grid, L, heads, nb, b, layout)
        for seed in range(20 if not rope else 8):
            simulate(its, seed, rope)
        for lag in range(5 if rope else 4):          # each role in turn falling behind
            for seed in range(3):
                simulate(its, seed, rope, lag=lag)


def test_model_catches_an_unrotated_q():
    """The checker itself: in the RoPE kernels an MMA that started an item on
    the landed Q (q_full) instead of the rotated one (q_ready) would let the
    producer reload the Q tiles while the rotating warps are still an item
    behind; the model must flag that (a parity wait that aliases, or a
    deadlock)."""
    its = items_for((3, 30, 40, 2, 3, 3), 0, 2, 3, 1, op.SHIFTED)
    global mma
    good_mma = mma

    def unrotated(src, rope):
        for op_ in good_mma(src, rope):
            yield ('wait', 'q_full', op_[2]) if op_[:2] == ('wait', 'q_ready') else op_
    mma = unrotated
    try:
        with pytest.raises((AssertionError, RuntimeError)):
            for seed in range(200):
                simulate(its, seed, rope=True, lag=4)      # the RoPE warps fall behind
    finally:
        mma = good_mma


class Dynamic:
    """One CTA's view of the global item counter: its producer draws the next
    index when it fills ring slot u, and its consumers read that slot."""
    def __init__(self, items, counter):
        self.items, self.counter, self.ring = items, counter, {}

    def draw(self, u):
        n = self.counter[0]
        self.counter[0] += 1
        self.ring[u] = self.items[n] if n < len(self.items) else None
        return self.ring[u]

    def get(self, u):
        return self.ring[u]


def simulate_grid(grid, L, heads, ncta, seed, layout=op.REGULAR, rope=False, slow=None):
    """Several CTAs at once, items drawn from one global counter in the
    kernel's order.  A CTA in `slow` is scheduled only when nothing else can
    move or with probability 1/20.  Checks: no deadlock, exact parity waits
    in every CTA, and every item drawn exactly once."""
    rnd = random.Random(seed)
    items = all_items(grid, L, heads, layout)
    need = counts(rope)
    counter = [0]
    roles, done, arr, srcs = [], {}, {}, []
    for c in range(ncta):
        src = Dynamic(items, counter)
        srcs.append(src)
        rs = [producer(src), mma(src, rope), softmax(src, 0), softmax(src, 1)]
        if rope: rs.append(rope_warps(src))
        roles += [(c, r) for r in rs]
        for b in need:
            done[(c, b)] = 0
            arr[(c, b)] = 0
    pending = [next(r, None) for _, r in roles]
    while any(p is not None for p in pending):
        ready = []
        for idx, op_ in enumerate(pending):
            if op_ is None: continue
            c = roles[idx][0]
            if op_[0] == 'wait':
                b, m = (c, op_[1]), op_[2]
                if (done[b] & 1) != (m & 1):
                    assert done[b] == m + 1, ("parity wait passes at the wrong phase", c, op_, done[b])
                    ready.append(idx)
            else:
                ready.append(idx)
        if not ready:
            raise RuntimeError("DEADLOCK: %s" % [(roles[i][0], p) for i, p in enumerate(pending) if p])
        if slow is not None and rnd.random() >= 0.05:
            fast = [i for i in ready if roles[i][0] not in slow]
            ready = fast or ready
        idx = rnd.choice(ready)
        c, op_ = roles[idx][0], pending[idx]
        if op_[0] in ('arrive', 'commit'):
            b = (c, op_[1])
            arr[b] += 1
            if arr[b] == need[op_[1]]:
                arr[b] = 0
                done[b] += 1
        pending[idx] = next(roles[idx][1], None)
    assert counter[0] == len(items) + ncta            # every item drawn once, one end mark per CTA
    drawn = sorted(it for s_ in srcs for it in s_.ring.values() if it is not None)
    assert drawn == sorted(items)


GRID_CASES = [((3, 30, 40, 2, 3, 3), 300, 2, 5), ((2, 45, 80, 1, 3, 3), 16, 3, 4),
              ((4, 40, 60, 2, 8, 8), 130, 2, 6), ((3, 9, 16, 1, 1, 1), 7, 2, 3)]


@pytest.mark.parametrize("layout", [op.REGULAR, op.SHIFTED])
@pytest.mark.parametrize("grid,L,heads,ncta", GRID_CASES)
def test_dynamic_items_across_ctas(grid, L, heads, ncta, layout):
    for seed in range(6):
        simulate_grid(grid, L, heads, ncta, seed, layout)
    for c in range(min(ncta, 3)):                      # each of a few CTAs falling behind
        simulate_grid(grid, L, heads, ncta, 100 + c, layout, slow={c})
    simulate_grid(grid, L, heads, ncta, 7, layout, rope=True)
