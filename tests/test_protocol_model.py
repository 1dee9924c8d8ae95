"""CPU model of the persistent attention kernel's barrier protocol.

The kernel (csrc/attn_tc.cu) coordinates a TMA producer, one MMA-issuing
thread and two softmax warpgroups through mbarriers that are waited on by
phase parity.  This model replays each role's sequence of waits, arrivals
and commits (a commit arrives when the MMAs before it finish; here, at once)
in random interleavings over real work-item lists, and checks that:
  * no interleaving deadlocks, and
  * every parity wait passes only at the phase it means: try_wait.parity(m&1)
    also passes when the barrier is one phase *behind* the target, or two
    ahead, so either would be a silent protocol error on the GPU.
The sequences mirror attn_tc_kernel's roles; a change to the kernel's
protocol must be made here too and checked before it runs on a GPU.
"""
import random

import numpy as np
import pytest

from oracle import plan as op

def items_for(grid, L, heads, nblocks, b, layout=op.REGULAR):
    """Work items (window, kv tiles, query tiles) that persistent CTA b walks."""
    BM=128
    out=[]
    off, _ = op.layout_tables(*grid, layout)
    sizes=np.diff(off); nwin=len(sizes)
    tt=(L+BM-1)//BM
    pairs=[]
    for w in range(nwin):
        vt=(sizes[w]+BM-1)//BM; nkv=vt+tt
        for jp in range((nkv+1)//2):
            pairs.append((w, nkv, min(2, nkv-2*jp)))
    items=[pairs[it % len(pairs)] for it in range(len(pairs)*heads)]
    return items[b::nblocks]

COUNT={'q_full':1,'q_empty':1,'pl_full0':1,'pl_full1':1,'pl_empty0':1,'pl_empty1':1,
       's_full0':1,'s_full1':1,'p_full0':1,'p_full1':1,'o_full0':1,'o_full1':1,
       'o_empty0':1,'o_empty1':1}

def producer(items):
    # payload e (global): item start -> [K(g0)]; step j -> [V(g0+j), K(g0+j+1)] (K only if
    # the item has tile j+1).  Payload e lives in slot e&1; it may load once payload e-2
    # is released (its tiles use the same K/V stages).
    e=0; k=0
    for (w,nkv,nq) in items:
        if k>0: yield ('wait','q_empty',k-1)
        yield ('arrive','q_full'); k+=1
        for p in range(nkv+1):
            if e>=2: yield ('wait','pl_empty%d'%(e&1),(e>>1)-1)
            yield ('arrive','pl_full%d'%(e&1))
            e+=1
def mma(items):
    e=0; k=0; cs=[0,0]; co=[0,0]
    for (w,nkv,nq) in items:
        yield ('wait','q_full',k)
        yield ('wait','pl_full%d'%(e&1),e>>1)          # payload [K(0)]
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

def softmax(items,i):
    cs=0; co=0
    for (w,nkv,nq) in items:
        if i>=nq: continue
        for j in range(nkv):
            yield ('wait','s_full%d'%i,cs+j)
            yield ('arrive','p_full%d'%i)
        cs+=nkv
        yield ('wait','o_full%d'%i,co)
        yield ('arrive','o_empty%d'%i); co+=1

def simulate(items, seed):
    rnd=random.Random(seed)
    done={b:0 for b in COUNT}
    roles=[producer(items),mma(items),softmax(items,0),softmax(items,1)]
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
        idx=rnd.choice(ready)
        op_=pending[idx]
        if op_[0] in ('arrive','commit'): done[op_[1]]+=1
        pending[idx]=next(roles[idx],None); steps+=1
    return steps

CASES = [((2, 45, 80, 1, 3, 3), 16, 2, 152), ((2, 45, 80, 1, 3, 3), 16, 2, 7), ((3, 30, 40, 2, 3, 3), 300, 2, 5),
         ((3, 30, 40, 2, 3, 3), 0, 2, 3), ((21, 68, 120, 4, 3, 3), 256, 1, 40), ((2, 45, 80, 1, 9, 16), 3, 2, 11),
         ((2, 3, 200, 1, 1, 9), 0, 1, 2)]


@pytest.mark.parametrize("layout", [op.REGULAR, op.SHIFTED])
@pytest.mark.parametrize("grid,L,heads,nb", CASES)
def test_protocol_has_no_deadlock_and_exact_parity(grid, L, heads, nb, layout):
    for b in range(min(nb, 4)):
        its = items_for(grid, L, heads, nb, b, layout)
        for seed in range(20):
            simulate(its, seed)
