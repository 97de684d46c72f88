"""Models of the tensor-core kernels' barrier protocols, run under random
interleavings on the CPU: the fused backward (bwd_main_kernel in
self_attention_backward_gb300/csrc/tc_bwd.cu), the two passes of the two-pass
mode on CTA pairs (bwd_kv_pair_kernel, bwd_q_pair_kernel in
self_attention_backward_gb300/csrc/tc_pair.cu) and the forward (fwd_kernel in
self_attention_backward_gb300/csrc/tc_fwd.cu).

Every role of one CTA is a coroutine that makes the same waits, arrivals, MMA
issues and commits, in the same order and with the same phase parities, as the
kernel: the TMA producer, the MMA issuer, the softmax warps (two warpgroups of
four warps), the four dQ drain warps and, for head_dim <= 32, the dQ issuer.
Each issuing thread's MMAs and commits go through its own FIFO and complete in
issue order; the two FIFOs interleave freely (the kernel relies on no order
between issuers).  mbarriers keep a completed-phase count and answer a parity
wait as the hardware does.

For many sub-tile counts and random schedules the model checks:
- every wait that passes sees exactly the phase it means (a ring or a parity
  test that could alias would pass a phase early or late);
- no arrival lands on a phase other than the barrier's current one;
- no data hazard: an MMA or a softmax warp reads a TMEM buffer, a Q/dO stage,
  a dS block or the dQ accumulator only when it holds the sub-tile (or group)
  the reader means, and nothing is overwritten before its last reader ran;
- no deadlock: every role finishes.
"""
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.done, self.arrived = name, count, 0, 0

    def passes(self, k):
        # try_wait.parity(k & 1): true once the phase with that parity completed
        return (self.done & 1) != (k & 1)

    def arrive(self, k):
        assert k == self.done, f"{self.name}: arrival for phase {k} while phase {self.done} is open"
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.done += 1


def run(nsub, split, NB, NST, seed, dqe_pair=True, with_dq=True, two_issuers=False, pf_ring=4, slow_role=None,
        sf_ring=None):
    """One random schedule of one CTA with nsub sub-tiles.  split: the dQ MMAs
    have an issuing thread of their own.  dqe_pair: the drain's "accumulator
    read" barrier alternates between two barriers by group parity, as the
    kernel does (False models a single barrier).  two_issuers: the fused
    kernel's two main issuing threads, one per sub-tile parity (each issues
    dV/dK(u) and then S/dP(u+NB) for its u, and the odd one first waits for
    dV/dK(0) to be done); pf_ring: the number of PF barriers.  slow_role: the
    index of a role the scheduler picks only rarely while others can run.
    with_dq=False models the two-pass mode's single-CTA dK/dV pass
    (bwd_dkdv_kernel): one issuer, no dQ, no drain, no dS ring."""
    rnd = random.Random(seed)
    ngrp = (nsub + 1) // 2
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    nsf = sf_ring or NB                     # SF barriers: a ring over the sub-tiles
    for b in range(nsf):
        bar(("SF", b))
    for x in range(pf_ring):
        bar(("PF", x), 4)           # four warps of one warpgroup
    for s in range(NST):
        bar(("QF", s))
        bar(("QE", s))
    for x in range(2 if dqe_pair else 1):
        bar(("DQE", x), 4)          # four drain warps

    def dqe(g):
        """The barrier and phase index on which group g's drain arrives."""
        return (bar(("DQE", g & 1)), g >> 1) if dqe_pair else (bar(("DQE", 0)), g)
    for x in range(2):
        bar(("DQF", x))

    # data state
    tmem = {b: ("free", None) for b in range(NB)}               # whole buffer, MMA side
    tq = {(b, q): None for b in range(NB) for q in range(4)}     # per lane quarter: ("S"|"P", u)
    stage = {s: None for s in range(NST)}                         # sub-tile loaded in stage s
    stage_readers = {s: set() for s in range(NST)}
    stage_soft = {s: 0 for s in range(NST)}                       # softmax warps done with the stage
    ds = {(blk, q): ("zero", None, True) for blk in range(4) for q in range(4)}  # (kind, u, read by dQ)
    acc = {q: ("idle", -1) for q in range(4)}                     # dQ accumulator per quarter
    fifo = {"main": [], "main1": [], "dq": []}
    dvdk_done = set()

    def mma_sdp(u):
        b, s = u % NB, u % NST
        assert tmem[b][0] == "free", f"S/dP({u}) overwrites buffer {b} holding {tmem[b]}"
        assert stage[s] == u, f"S/dP({u}) reads stage {s} holding {stage[s]}"
        stage_readers[s].add("sdp")
        tmem[b] = ("S", u)
        for q in range(4):
            tq[(b, q)] = ("S", u)

    def mma_dvdk(u):
        b, s = u % NB, u % NST
        # the first dV/dK product overwrites the accumulators; every later one adds
        assert u == 0 or 0 in dvdk_done, f"dV/dK({u}) adds to accumulators dV/dK(0) has not yet zeroed"
        dvdk_done.add(u)
        for q in range(4):
            assert tq[(b, q)] == ("P", u), f"dV/dK({u}) reads {tq[(b, q)]}"
        assert stage[s] == u and "sdp" in stage_readers[s]
        stage_readers[s].add("dvdk")
        tmem[b] = ("free", None)

    def mma_dq(g):
        for j in (2 * g, 2 * g + 1):
            if j >= nsub:
                continue
            for q in range(4):
                kind, uu, _ = ds[(j & 3, q)]
                assert (kind, uu) == ("dS", j), f"dQ({g}) reads dS block {j & 3} holding {(kind, uu)}"
                ds[(j & 3, q)] = ("dS", j, True)
        for q in range(4):
            assert acc[q] in (("idle", -1), ("read", g - 1)), f"dQ({g}) overwrites accumulator {acc[q]}"
            acc[q] = ("dq", g)

    def issue(who, item):
        fifo[who].append(item)

    # ---------------------------------------------------------------- roles
    def producer():
        for u in range(nsub):
            s = u % NST
            k = u // NST - 1
            yield ("wait", bar(("QE", s)), k)
            if stage[s] is not None:
                assert stage_readers[s] >= {"sdp", "dvdk"} and stage_soft[s] == 4, \
                    f"stage {s} reused early: {stage_readers[s]}, {stage_soft[s]} softmax warps done"
            stage[s] = u
            stage_readers[s] = set()
            stage_soft[s] = 0
            yield ("arrive", bar(("QF", s)), u // NST)

    def main_issuer(par=0, step=1):
        me = "main" if par == 0 else "main1"
        if par == 0:
            for u in range(min(NB, nsub)):
                yield ("wait", bar(("QF", u)), 0)
            for u in range(min(NB, nsub)):
                issue(me, ("mma", mma_sdp, u))
                issue(me, ("commit", bar(("SF", u % nsf)), u // nsf))
        elif nsub > 1:
            yield ("wait", bar(("QE", 0)), 0)
        for u in range(par, nsub, step):
            yield ("wait", bar(("PF", u % pf_ring)), u // pf_ring)
            issue(me, ("mma", mma_dvdk, u))
            issue(me, ("commit", bar(("QE", u % NST)), u // NST))
            if with_dq and not split and (u % 2 == 1 or u == nsub - 1):
                g = u // 2
                issue(me, ("mma", mma_dq, g))
                issue(me, ("commit", bar(("DQF", g & 1)), g >> 1))
            if u + NB < nsub:
                v = u + NB
                issue(me, ("mma", mma_sdp, v))
                issue(me, ("commit", bar(("SF", v % nsf)), v // nsf))

    def softmax(grp, q):
        if grp < nsub:
            yield ("wait", bar(("QF", grp % NST)), grp // NST)
            assert stage[grp % NST] == grp, f"softmax reads the statistics of stage {grp % NST} too early"
        for u in range(grp, nsub, 2):
            b, s = u % NB, u % NST
            # the statistics of u were read at the end of u-2 (or before the loop)
            yield ("wait", bar(("SF", u % nsf)), u // nsf)
            if with_dq and split and u >= 4:
                h = (u - 4) >> 1
                yield ("wait", bar(("DQF", h & 1)), h >> 1)
            # the warp's work: TMEM S/dP(u) -> P/dS(u); dS into the ring
            assert tq[(b, q)] == ("S", u), f"softmax({u}) reads {tq[(b, q)]}"
            assert stage[s] == u
            if with_dq:
                kind, uu, read = ds[(u & 3, q)]
                assert read, f"softmax({u}) overwrites dS of sub-tile {uu} before its dQ product read it"
                ds[(u & 3, q)] = ("dS", u, False)
            tq[(b, q)] = ("P", u)
            stage_soft[s] += 1
            if u + NB < nsub:
                v = u + NB
                yield ("wait", bar(("QF", v % NST)), v // NST)
            if u + 2 < nsub:
                yield ("wait", bar(("QF", (u + 2) % NST)), (u + 2) // NST)
            if with_dq and not split and (u % 2 == 1 or u == nsub - 1) and u >= 2:
                yield ("wait",) + dqe((u >> 1) - 1)
            if u + 2 < nsub:
                # the next sub-tile's statistics are read before PF(u)
                assert stage[(u + 2) % NST] == u + 2, f"softmax({u}) reads stage {(u + 2) % NST} too early"
            yield ("arrive", bar(("PF", u % pf_ring)), u // pf_ring)

    def dq_issuer():
        for g in range(ngrp):
            for u in (2 * g, 2 * g + 1):
                if u < nsub:
                    yield ("wait", bar(("PF", u % pf_ring)), u // pf_ring)
            if g > 0:
                yield ("wait",) + dqe(g - 1)
            issue("dq", ("mma", mma_dq, g))
            issue("dq", ("commit", bar(("DQF", g & 1)), g >> 1))

    def drain(q):
        for g in range(ngrp):
            yield ("wait", bar(("DQF", g & 1)), g >> 1)
            assert acc[q] == ("dq", g), f"drain({g}) reads {acc[q]}"
            acc[q] = ("read", g)
            yield ("arrive",) + dqe(g)

    roles = [producer()]
    roles += [main_issuer(0, 2), main_issuer(1, 2)] if two_issuers else [main_issuer()]
    roles += [softmax(g, q) for g in range(2) for q in range(4)]
    if with_dq:
        roles += [drain(q) for q in range(4)]
        if split:
            roles.append(dq_issuer())
    pending = {i: None for i in range(len(roles))}   # the request each role is blocked on

    def advance(i):
        try:
            pending[i] = roles[i].send(None)
        except StopIteration:
            pending[i] = "done"

    for i in range(len(roles)):
        advance(i)
    steps = 0
    while True:
        steps += 1
        assert steps < 200000
        enabled = []
        for i, req in pending.items():
            if req == "done":
                continue
            kind = req[0]
            if kind == "wait":
                _, br, k = req
                # a later phase completed before this waiter saw its own: on the
                # GPU the parity test could then block forever or pass a phase late
                assert br.done <= k + 1, f"{br.name}: phase {k + 1} completed before a waiter for phase {k} passed"
                if br.passes(k):
                    enabled.append(("role", i))
            else:
                enabled.append(("role", i))
        for who in ("main", "main1", "dq"):
            if fifo[who]:
                enabled.append(("pipe", who))
        if not enabled:
            blocked = {i: (r[1].name, r[2], r[1].done) for i, r in pending.items() if r != "done"}
            assert not blocked, f"deadlock: {blocked}"
            assert not any(fifo.values())
            return
        if slow_role is not None and len(enabled) > 1 and rnd.random() > 0.02:
            # a role index, or the name of an issuing thread's MMA pipe
            slow = ("pipe", slow_role) if isinstance(slow_role, str) else ("role", slow_role)
            enabled = [e for e in enabled if e != slow] or enabled
        kind, x = rnd.choice(enabled)
        if kind == "pipe":
            item = fifo[x].pop(0)
            if item[0] == "mma":
                item[1](item[2])
            else:
                item[1].arrive(item[2])
            continue
        req = pending[x]
        if req[0] == "wait":
            _, br, k = req
            assert br.done == k + 1, f"{br.name}: wait for phase {k} passed at {br.done} completed phases"
        elif req[0] == "arrive":
            req[1].arrive(req[2])
        advance(x)


def run_fused(nsub, NB, NST, seed, two_issuers, pf_ring=8, sf_ring=None, slow_role=None, s_first=True,
              plant=None):
    """One random schedule of one CTA of the fused backward kernel (bwd_main_kernel).

    Roles: the TMA producer (stage s of sub-tile u after QE(s)); one or two main
    issuers (two: one per sub-tile parity); four softmax warps in each of two
    warpgroups (even / odd sub-tiles); the dQ issuer; four drain warps.  Buffer
    b = u % NB has an S^T region and a dP^T region.  After PF(u) the issuer of
    u issues, in this order, dV(u) (reads P(u) from the S region), S^T(u+NB)
    (overwrites the S region) and commits SFs(u+NB), dK(u) (reads dS(u) from
    the dP region), commits QE, dP^T(u+NB) (overwrites the dP region) and
    commits SFd(u+NB).  The softmax of u waits SFs(u) (and the dQ product that
    last read its dS ring block), turns S into P, waits SFd(u), turns dP into
    dS (region and ring), waits for the stages of u+NB and u+2, reads the
    statistics of u+2 and arrives PF(u).  s_first=False issues dV/dK(u) before
    both halves of S/dP(u+NB).  plant
    names a mistake to put into the protocol: "no_dqf_wait" drops the softmax's
    wait for the dQ product, "s_before_dv" issues S^T(u+NB) before dV(u)."""
    rnd = random.Random(seed)
    ngrp = (nsub + 1) // 2
    nsf = sf_ring or 2 * NB
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    for b in range(nsf):
        bar(("SFs", b))
        bar(("SFd", b))
    for x in range(pf_ring):
        bar(("PF", x), 4)
    for st in range(NST):
        bar(("QF", st))
        bar(("QE", st))
    for x in range(2):
        bar(("DQE", x), 4)
        bar(("DQF", x))

    sreg = {(b, q): ("free", None) for b in range(NB) for q in range(4)}
    dreg = {(b, q): ("free", None) for b in range(NB) for q in range(4)}
    stage = {st: None for st in range(NST)}
    readers = {st: set() for st in range(NST)}
    stage_soft = {st: 0 for st in range(NST)}
    ds = {(blk, q): ("zero", None, True) for blk in range(4) for q in range(4)}
    acc = {q: ("idle", -1) for q in range(4)}
    fifo = {"main": [], "main1": [], "dq": []}
    dv_done = set()

    def check_stage(u, what):
        st = u % NST
        assert stage[st] == u, f"{what}({u}) reads stage {st} holding {stage[st]}"
        readers[st].add(what)

    def mma_s(u):
        b = u % NB
        for q in range(4):
            assert sreg[(b, q)][0] == "free", f"S({u}) overwrites {sreg[(b, q)]}"
            sreg[(b, q)] = ("S", u)
        check_stage(u, "s")

    def mma_dp(u):
        b = u % NB
        for q in range(4):
            assert dreg[(b, q)][0] == "free", f"dP({u}) overwrites {dreg[(b, q)]}"
            dreg[(b, q)] = ("dP", u)
        check_stage(u, "dp")

    def mma_dv(u):
        b = u % NB
        assert u == 0 or 0 in dv_done, f"dV({u}) adds to accumulators dV(0) has not yet zeroed"
        dv_done.add(u)
        for q in range(4):
            assert sreg[(b, q)] == ("P", u), f"dV({u}) reads {sreg[(b, q)]}"
            sreg[(b, q)] = ("free", None)
        check_stage(u, "dv")

    def mma_dk(u):
        b = u % NB
        for q in range(4):
            assert dreg[(b, q)] == ("dS", u), f"dK({u}) reads {dreg[(b, q)]}"
            dreg[(b, q)] = ("free", None)
        check_stage(u, "dk")

    def mma_dq(g):
        for j in (2 * g, 2 * g + 1):
            if j >= nsub:
                continue
            for q in range(4):
                kind, uu, _ = ds[(j & 3, q)]
                assert (kind, uu) == ("dS", j), f"dQ({g}) reads dS block {j & 3} holding {(kind, uu)}"
                ds[(j & 3, q)] = ("dS", j, True)
        for q in range(4):
            assert acc[q] in (("idle", -1), ("read", g - 1)), f"dQ({g}) overwrites accumulator {acc[q]}"
            acc[q] = ("dq", g)

    def producer():
        for u in range(nsub):
            st = u % NST
            yield ("wait", bar(("QE", st)), u // NST - 1)
            if stage[st] is not None:
                assert readers[st] >= {"s", "dp", "dv", "dk"} and stage_soft[st] == 4, \
                    f"stage {st} reused early: {readers[st]}, {stage_soft[st]} softmax warps done"
            stage[st] = u
            readers[st] = set()
            stage_soft[st] = 0
            yield ("arrive", bar(("QF", st)), u // NST)

    def issue_sdp(me, v, split):
        fifo[me].append(("mma", mma_s, v))
        fifo[me].append(("commit", bar(("SFs", v % nsf)), v // nsf))
        if not split:
            fifo[me].append(("mma", mma_dp, v))
            fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))

    def main_issuer(par, step):
        me = "main" if par == 0 else "main1"
        if par == 0:
            for u in range(min(NB, nsub)):
                yield ("wait", bar(("QF", u)), 0)
            for u in range(min(NB, nsub)):
                issue_sdp(me, u, False)
        elif nsub > 1:
            yield ("wait", bar(("QE", 0)), 0)
        for u in range(par, nsub, step):
            yield ("wait", bar(("PF", u % pf_ring)), u // pf_ring)
            v = u + NB
            if plant != "s_before_dv":
                fifo[me].append(("mma", mma_dv, u))
            if s_first and v < nsub:
                fifo[me].append(("mma", mma_s, v))
                fifo[me].append(("commit", bar(("SFs", v % nsf)), v // nsf))
            if plant == "s_before_dv":
                fifo[me].append(("mma", mma_dv, u))
            fifo[me].append(("mma", mma_dk, u))
            fifo[me].append(("commit", bar(("QE", u % NST)), u // NST))
            if v < nsub:
                if not s_first:
                    fifo[me].append(("mma", mma_s, v))
                    fifo[me].append(("commit", bar(("SFs", v % nsf)), v // nsf))
                fifo[me].append(("mma", mma_dp, v))
                fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))

    def softmax(grp, q):
        if grp < nsub:
            yield ("wait", bar(("QF", grp % NST)), grp // NST)
            assert stage[grp % NST] == grp
        for u in range(grp, nsub, 2):
            b, st = u % NB, u % NST
            yield ("wait", bar(("SFs", u % nsf)), u // nsf)
            if u >= 4 and plant != "no_dqf_wait":
                h = (u - 4) >> 1
                yield ("wait", bar(("DQF", h & 1)), h >> 1)
            assert sreg[(b, q)] == ("S", u), f"softmax({u}) reads S region {sreg[(b, q)]}"
            sreg[(b, q)] = ("P", u)
            yield ("wait", bar(("SFd", u % nsf)), u // nsf)
            assert dreg[(b, q)] == ("dP", u), f"softmax({u}) reads dP region {dreg[(b, q)]}"
            dreg[(b, q)] = ("dS", u)
            kind, uu, read = ds[(u & 3, q)]
            assert read, f"softmax({u}) overwrites dS of sub-tile {uu} before its dQ product read it"
            ds[(u & 3, q)] = ("dS", u, False)
            stage_soft[st] += 1
            if u + NB < nsub:
                v = u + NB
                yield ("wait", bar(("QF", v % NST)), v // NST)
            if u + 2 < nsub:
                yield ("wait", bar(("QF", (u + 2) % NST)), (u + 2) // NST)
                assert stage[(u + 2) % NST] == u + 2
            yield ("arrive", bar(("PF", u % pf_ring)), u // pf_ring)

    def dq_issuer():
        for g in range(ngrp):
            for u in (2 * g, 2 * g + 1):
                if u < nsub:
                    yield ("wait", bar(("PF", u % pf_ring)), u // pf_ring)
            if g > 0:
                yield ("wait", bar(("DQE", (g - 1) & 1)), (g - 1) >> 1)
            fifo["dq"].append(("mma", mma_dq, g))
            fifo["dq"].append(("commit", bar(("DQF", g & 1)), g >> 1))

    def drain(q):
        for g in range(ngrp):
            yield ("wait", bar(("DQF", g & 1)), g >> 1)
            assert acc[q] == ("dq", g), f"drain({g}) reads {acc[q]}"
            acc[q] = ("read", g)
            yield ("arrive", bar(("DQE", g & 1)), g >> 1)

    roles = [producer()]
    roles += [main_issuer(0, 2), main_issuer(1, 2)] if two_issuers else [main_issuer(0, 1)]
    roles += [softmax(g, q) for g in range(2) for q in range(4)]
    roles += [drain(q) for q in range(4)] + [dq_issuer()]
    schedule(roles, fifo, rnd, slow_role)


def run_persistent(items, NB, NST, seed, two_issuers, pf_ring=8, slow_role=None, plant=None, kvbuf=1,
                   ds_smem=False, dk_first=False, dse_by_qe=False, p_ready=False, lag=False, by_kind=False):
    """One random schedule of one persistent CTA of the fused backward kernel
    walking several work items (units or pieces) in turn; items lists their
    sub-tile counts.  Sub-tiles U and 128-query groups G are numbered across
    the CTA's items, and every ring (Q/dO stages, S/dP buffers, S^T / dP^T
    barriers, PF, dS ring blocks 2 (G & 1) + s, dQ barriers) runs on those
    numbers; each item has its own K/V tile and dV/dK accumulators.

    Roles as in run_fused, plus: the producer, per item the K/V tile into
    buffer i % kvbuf after KVE of item i - kvbuf (which the dQ issuer commits,
    on that buffer's barrier, after the item's last dQ product), then the
    item's Q/dO stages; main issuers of global parity (the one of
    parity 0 issues each item's first min(NB, nsub) S/dP products, after the
    other issuer's last dV/dK of the previous item (that sub-tile's QE commit),
    the item's K/V (KV) and stages; before an item's first dV/dK each issuer waits for the previous
    item's epilogue (EPI), and the issuer that does not own the item's first
    sub-tile also for dV/dK of that sub-tile; each commits ACC per item); the
    drain warps run each item's epilogue (ACC waits, accumulator reads, EPI
    arrive).  ds_smem: dK(u) reads dS(u) from its shared-memory ring block
    (as the dQ product does), so the softmax leaves the dP region free once it
    has read dP(u); the issuer issues dV(u), S/dP(u+NB), then dK(u) and commits
    QE and DSE of the block (dk_first: dV(u), S(u+NB), dK(u) and its commits,
    dP(u+NB)), and the softmax waits for the DSE of the block's
    previous sub-tile before writing it (else the older form: dS(u) also in
    the dP region, read there by dK(u), which precedes dP(u+NB)).
    dse_by_qe (with ds_smem and dk_first): no DSE barriers; with its S^T wait
    the softmax of the item's sub-tile ul >= 4 waits for QE of sub-tile u-4,
    the block's previous sub-tile (the item's groups before its last are
    full).  For ul < 4 the previous sub-tile is in an earlier item, whose dK
    products are all done before S(u) is: the prologue waits for the other
    issuer's last ACCB and follows its own thread's dK products, and every
    later S/dP of the item follows a PF of the item.
    p_ready: the softmax also arrives PR(u), a ring like PF, once P(u) is
    written and the stage of u+NB is loaded; the issuer waits PR(u) for dV(u)
    and S(u+NB), then PF(u) for dK(u) and dP(u+NB).  lag (with p_ready): the
    issuer waits only PR(u), then issues dV(u), S(u+NB) and the dK / dP of its
    previous sub-tile of the item (u-2: its PF came from the same warpgroup
    before PR(u)); after the item's last it waits PF for the pending one.
    by_kind (with p_ready): the two issuers split the work by MMA kind, not
    by sub-tile parity: issuer A ("main") takes every sub-tile's dV(u) and
    S(u+NB) after PR(u), issuer B ("main1") its dK(u) and dP(u+NB) after
    PF(u), each also the item prologue's S (A) or dP (B) products; a stage is
    free once both have committed QE (a barrier of two arrivals), and each
    commits ACC (A) or ACCB (B) every item.  plant:
    "no_epi_wait" drops the issuers' EPI wait; "no_kve_wait" lets the K/V
    producer skip KVE; "no_dse_wait" drops the softmax's DSE wait;
    "accb_prologue" makes the prologue wait for the other issuer's ACCB
    instead of its last QE."""
    rnd = random.Random(seed)
    nsf = 2 * NB
    UT = sum(items)
    item_of, ul_of = [], []
    for it, n in enumerate(items):
        item_of += [it] * n
        ul_of += list(range(n))
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    for b in range(nsf):
        bar(("SFs", b))
        bar(("SFd", b))
    for x in range(pf_ring):
        bar(("PF", x), 4)
        bar(("PR", x), 4)
    for st in range(NST):
        bar(("QF", st))
        bar(("QE", st), 2 if by_kind else 1)
    for x in range(2):
        bar(("DQE", x), 4)
        bar(("DQF", x))
    for b in range(kvbuf):
        bar(("KV", b))
        bar(("KVE", b))
    bar("ACC")
    bar("ACCB")
    bar("EPI", 4)
    for b in range(4):
        bar(("DSE", b))
    # dS ring block of each sub-tile (2 (G & 1) + its place in the group) and
    # which use of that block it is
    blk_of, use_of, uses, g0 = [], [], [0] * 4, 0
    for n in items:
        for ul in range(n):
            b = 2 * ((g0 + ul // 2) & 1) + (ul & 1)
            blk_of.append(b)
            use_of.append(uses[b])
            uses[b] += 1
        g0 += (n + 1) // 2
    ds_readers = {"dq", "dk"} if ds_smem else {"dq"}

    sreg = {(b, q): ("free", None) for b in range(NB) for q in range(4)}
    dreg = {(b, q): ("free", None) for b in range(NB) for q in range(4)}
    stage = {st: None for st in range(NST)}
    readers = {st: set() for st in range(NST)}
    stage_soft = {st: 0 for st in range(NST)}
    ds = {(blk, q): ("zero", None, {"dq", "dk"}) for blk in range(4) for q in range(4)}
    acc = {q: ("idle", -1) for q in range(4)}
    kv = [None] * kvbuf
    kv_reads = {it: 0 for it in range(len(items))}       # S, dP and dQ products of the item executed
    ready_for = {q: None for q in range(4)}              # item whose products a lane quarter's accumulators await
    counts = {}
    fifo = {"main": [], "main1": [], "dq": []}

    def check_stage(u, what):
        st = u % NST
        assert stage[st] == u, f"{what}({u}) reads stage {st} holding {stage[st]}"
        readers[st].add(what)

    def check_kv(u, what):
        it = item_of[u]
        assert kv[it % kvbuf] == it, f"{what}({u}) of item {it} reads K/V of item {kv[it % kvbuf]}"

    def mma_s(u):
        b = u % NB
        for q in range(4):
            assert sreg[(b, q)][0] == "free", f"S({u}) overwrites {sreg[(b, q)]}"
            sreg[(b, q)] = ("S", u)
        check_stage(u, "s")
        check_kv(u, "S")
        kv_reads[item_of[u]] += 1

    def mma_dp(u):
        b = u % NB
        for q in range(4):
            assert dreg[(b, q)][0] == "free", f"dP({u}) overwrites {dreg[(b, q)]}"
            dreg[(b, q)] = ("dP", u)
        check_stage(u, "dp")
        check_kv(u, "dP")
        kv_reads[item_of[u]] += 1

    def acc_use(u, what):
        # every dV/dK product accumulates; the drain zeroes the accumulators
        # (each warp its lane quarter) before an item and after its epilogue
        it = item_of[u]
        for q in range(4):
            assert ready_for[q] == it, \
                f"{what}({u}) of item {it} adds to accumulators quarter {q} holds for item {ready_for[q]}"
        counts[(it, what)] = counts.get((it, what), 0) + 1

    def mma_dv(u):
        b = u % NB
        acc_use(u, "dv")
        for q in range(4):
            assert sreg[(b, q)] == ("P", u), f"dV({u}) reads {sreg[(b, q)]}"
            sreg[(b, q)] = ("free", None)
        check_stage(u, "dv")

    def mma_dk(u):
        b = u % NB
        acc_use(u, "dk")
        for q in range(4):
            if ds_smem:
                kind, uu, rd = ds[(blk_of[u], q)]
                assert (kind, uu) == ("dS", u), f"dK({u}) reads dS block {blk_of[u]} holding {(kind, uu)}"
                ds[(blk_of[u], q)] = (kind, uu, rd | {"dk"})
            else:
                assert dreg[(b, q)] == ("dS", u), f"dK({u}) reads {dreg[(b, q)]}"
                dreg[(b, q)] = ("free", None)
        check_stage(u, "dk")

    def mma_dq(arg):
        g, us = arg
        for s_, u in enumerate(us):
            blk = 2 * (g & 1) + s_
            for q in range(4):
                kind, uu, rd = ds[(blk, q)]
                assert (kind, uu) == ("dS", u), f"dQ({g}) reads dS block {blk} holding {(kind, uu)}"
                ds[(blk, q)] = ("dS", u, rd | {"dq"})
            check_kv(u, "dQ")
        kv_reads[item_of[us[0]]] += 1
        for q in range(4):
            assert acc[q] in (("idle", -1), ("read", g - 1)), f"dQ({g}) overwrites accumulator {acc[q]}"
            acc[q] = ("dq", g)

    def producer():
        u = 0
        for it, n in enumerate(items):
            b = it % kvbuf
            if it >= kvbuf:
                if plant != "no_kve_wait":
                    yield ("wait", bar(("KVE", b)), it // kvbuf - 1)
                prev = items[it - kvbuf]
                assert kv_reads[it - kvbuf] == 2 * prev + (prev + 1) // 2, \
                    f"K/V of item {it} loaded while item {it - kvbuf} still reads its tile"
            kv[b] = it
            yield ("arrive", bar(("KV", b)), it // kvbuf)
            for _ in range(n):
                st = u % NST
                yield ("wait", bar(("QE", st)), u // NST - 1)
                if stage[st] is not None:
                    assert readers[st] >= {"s", "dp", "dv", "dk"} and stage_soft[st] == 4, \
                        f"stage {st} reused early: {readers[st]}, {stage_soft[st]} softmax warps done"
                stage[st] = u
                readers[st] = set()
                stage_soft[st] = 0
                yield ("arrive", bar(("QF", st)), u // NST)
                u += 1

    def issue_sdp(me, v):
        fifo[me].append(("mma", mma_s, v))
        fifo[me].append(("commit", bar(("SFs", v % nsf)), v // nsf))
        fifo[me].append(("mma", mma_dp, v))
        fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))

    # ACCB phases: one per item in which the odd issuer has a sub-tile
    odd_items = [it for it, n in enumerate(items)
                 if any((u % 2) == 1 for u in range(sum(items[:it]), sum(items[:it]) + n))]

    def issue_dkdp(me, pend):
        # dK(u) and, within the item, dP(u+NB), with their commits (the lag form
        # of the ring-dS, dK-first order)
        u, ul, n = pend
        v = u + NB
        fifo[me].append(("mma", mma_dk, u))
        fifo[me].append(("commit", bar(("QE", u % NST)), u // NST))
        if ds_smem and not dse_by_qe:
            fifo[me].append(("commit", bar(("DSE", blk_of[u])), use_of[u]))
        if ul + NB < n:
            fifo[me].append(("mma", mma_dp, v))
            fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))

    def kind_issuer(kind):
        # by_kind: A (kind 0) dV and S, B (kind 1) dK and dP
        me = "main" if kind == 0 else "main1"
        u0 = 0
        for it, n in enumerate(items):
            yield ("wait", bar(("KV", it % kvbuf)), it // kvbuf)
            for j in range(min(NB, n)):
                yield ("wait", bar(("QF", (u0 + j) % NST)), (u0 + j) // NST)
            for j in range(min(NB, n)):
                v = u0 + j
                if kind == 0:
                    fifo[me].append(("mma", mma_s, v))
                    fifo[me].append(("commit", bar(("SFs", v % nsf)), v // nsf))
                else:
                    fifo[me].append(("mma", mma_dp, v))
                    fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))
            first = True
            for ul in range(n):
                u = u0 + ul
                yield ("wait", bar(("PR" if kind == 0 else "PF", u % pf_ring)), u // pf_ring)
                if first:
                    if plant != "no_epi_wait":
                        yield ("wait", bar("EPI"), it)
                    first = False
                v = u + NB
                if kind == 0:
                    fifo[me].append(("mma", mma_dv, u))
                    fifo[me].append(("commit", bar(("QE", u % NST)), u // NST))
                    if ul + NB < n:
                        fifo[me].append(("mma", mma_s, v))
                        fifo[me].append(("commit", bar(("SFs", v % nsf)), v // nsf))
                else:
                    fifo[me].append(("mma", mma_dk, u))
                    fifo[me].append(("commit", bar(("QE", u % NST)), u // NST))
                    if ul + NB < n:
                        fifo[me].append(("mma", mma_dp, v))
                        fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))
            if first and plant != "no_epi_wait":
                yield ("wait", bar("EPI"), it)
            fifo[me].append(("commit", bar("ACC" if kind == 0 else "ACCB"), it))
            u0 += n

    def main_issuer(par):
        me = "main" if par == 0 else "main1"
        u0 = 0
        for it, n in enumerate(items):
            if par == 0:
                if it > 0 and two_issuers and plant == "accb_prologue":
                    yield ("wait", bar("ACCB"), it - 1)
                elif it > 0 and two_issuers and plant == "qe_prologue":
                    # the other issuer's last dK of the previous item (its QE commit):
                    # with 4 stages that barrier can be two phases behind
                    odd = [u for u in range(u0 - items[it - 1], u0) if u % 2 == 1]
                    if odd:
                        yield ("wait", bar(("QE", odd[-1] % NST)), odd[-1] // NST)
                elif it > 0 and two_issuers:
                    # the other issuer's latest ACCB phase: all its MMAs so far
                    # (the buffers' last readers among them) are done
                    kb = sum(1 for x in odd_items if x < it)
                    if kb:
                        yield ("wait", bar("ACCB"), kb - 1)
                yield ("wait", bar(("KV", it % kvbuf)), it // kvbuf)
                for j in range(min(NB, n)):
                    yield ("wait", bar(("QF", (u0 + j) % NST)), (u0 + j) // NST)
                for j in range(min(NB, n)):
                    issue_sdp(me, u0 + j)
            first = True
            pending = None
            for ul in range(n):
                u = u0 + ul
                if two_issuers and u % 2 != par:
                    continue
                yield ("wait", bar(("PR" if p_ready else "PF", u % pf_ring)), u // pf_ring)
                if first:
                    # the accumulators are zeroed for this item (EPI phase 0: at
                    # the start; phase i + 1: after item i's epilogue)
                    if plant != "no_epi_wait":
                        yield ("wait", bar("EPI"), it)
                    first = False
                v = u + NB
                fifo[me].append(("mma", mma_dv, u))
                if ul + NB < n:
                    fifo[me].append(("mma", mma_s, v))
                    fifo[me].append(("commit", bar(("SFs", v % nsf)), v // nsf))
                if p_ready and lag:
                    if pending is not None:
                        issue_dkdp(me, pending)
                    pending = (u, ul, n)
                    continue
                if p_ready and plant != "no_pf_after_pr":
                    yield ("wait", bar(("PF", u % pf_ring)), u // pf_ring)
                if ds_smem:
                    if ul + NB < n and not dk_first:
                        fifo[me].append(("mma", mma_dp, v))
                        fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))
                    fifo[me].append(("mma", mma_dk, u))
                    fifo[me].append(("commit", bar(("QE", u % NST)), u // NST))
                    if not dse_by_qe:
                        fifo[me].append(("commit", bar(("DSE", blk_of[u])), use_of[u]))
                    if ul + NB < n and dk_first:
                        fifo[me].append(("mma", mma_dp, v))
                        fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))
                    continue
                fifo[me].append(("mma", mma_dk, u))
                fifo[me].append(("commit", bar(("QE", u % NST)), u // NST))
                if ul + NB < n:
                    fifo[me].append(("mma", mma_dp, v))
                    fifo[me].append(("commit", bar(("SFd", v % nsf)), v // nsf))
            if pending is not None:
                pu = pending[0]
                if plant != "lag_no_final_pf":
                    yield ("wait", bar(("PF", pu % pf_ring)), pu // pf_ring)
                issue_dkdp(me, pending)
                pending = None
            if par == 0:
                # ACC every item: an issuer without a sub-tile first waits for the
                # zeroing for this item, so its phases keep in step with the drain's
                if first and plant != "no_epi_wait":
                    yield ("wait", bar("EPI"), it)
                fifo[me].append(("commit", bar("ACC"), it))
            elif plant == "accb_prologue":
                # (the aliasing form: an ACCB commit every item)
                if first:
                    yield ("wait", bar("EPI"), it)
                fifo[me].append(("commit", bar("ACCB"), it))
            elif not first:
                # ACCB only for items with a sub-tile of this issuer
                fifo[me].append(("commit", bar("ACCB"), odd_items.index(it)))
            u0 += n

    def softmax(grp, q):
        if grp < UT:
            yield ("wait", bar(("QF", grp % NST)), grp // NST)
            assert stage[grp % NST] == grp
        u0 = g0 = 0
        for it, n in enumerate(items):
            for ul in range(n):
                u = u0 + ul
                if u % 2 != grp:
                    continue
                g, s_ = g0 + ul // 2, ul & 1
                b, st, blk = u % NB, u % NST, 2 * (g & 1) + s_
                if ul < 2 and u != grp:
                    # the first sub-tile of a later item: statistics not fetched ahead
                    yield ("wait", bar(("QF", st)), u // NST)
                    assert stage[st] == u
                yield ("wait", bar(("SFs", u % nsf)), u // nsf)
                if g >= 2:
                    yield ("wait", bar(("DQF", (g - 2) & 1)), (g - 2) >> 1)
                if ds_smem and not dse_by_qe and use_of[u] > 0 and plant != "no_dse_wait":
                    # dK of the block's previous sub-tile is done with it
                    yield ("wait", bar(("DSE", blk)), use_of[u] - 1)
                if dse_by_qe and ul >= 4 and plant != "no_dse_wait":
                    yield ("wait", bar(("QE", (u - 4) % NST)), (u - 4) // NST)
                assert sreg[(b, q)] == ("S", u), f"softmax({u}) reads S region {sreg[(b, q)]}"
                sreg[(b, q)] = ("P", u)
                if p_ready:
                    # PR(u) certifies, as PF(u) does otherwise, that the stage of
                    # u+NB is loaded (S(u+NB) follows it)
                    if ul + NB < n and plant != "pr_without_stage":
                        v = u + NB
                        yield ("wait", bar(("QF", v % NST)), v // NST)
                    yield ("arrive", bar(("PR", u % pf_ring)), u // pf_ring)
                yield ("wait", bar(("SFd", u % nsf)), u // nsf)
                assert dreg[(b, q)] == ("dP", u), f"softmax({u}) reads dP region {dreg[(b, q)]}"
                dreg[(b, q)] = ("free", None) if ds_smem else ("dS", u)
                kind, uu, rd = ds[(blk, q)]
                assert rd >= ds_readers, \
                    f"softmax({u}) overwrites dS of sub-tile {uu} before its {sorted(ds_readers - rd)} product read it"
                ds[(blk, q)] = ("dS", u, set())
                stage_soft[st] += 1
                if ul + NB < n and not p_ready:
                    v = u + NB
                    yield ("wait", bar(("QF", v % NST)), v // NST)
                if ul + 2 < n:
                    yield ("wait", bar(("QF", (u + 2) % NST)), (u + 2) // NST)
                    assert stage[(u + 2) % NST] == u + 2
                yield ("arrive", bar(("PF", u % pf_ring)), u // pf_ring)
            u0 += n
            g0 += (n + 1) // 2

    def dq_issuer():
        u0 = g0 = 0
        for it, n in enumerate(items):
            for gl in range((n + 1) // 2):
                g = g0 + gl
                us = [u for u in (u0 + 2 * gl, u0 + 2 * gl + 1) if u < u0 + n]
                for u in us:
                    yield ("wait", bar(("PF", u % pf_ring)), u // pf_ring)
                if g > 0:
                    yield ("wait", bar(("DQE", (g - 1) & 1)), (g - 1) >> 1)
                fifo["dq"].append(("mma", mma_dq, (g, us)))
                fifo["dq"].append(("commit", bar(("DQF", g & 1)), g >> 1))
            fifo["dq"].append(("commit", bar(("KVE", it % kvbuf)), it // kvbuf))
            u0 += n
            g0 += (n + 1) // 2

    def drain(q):
        ready_for[q] = 0                                  # zeroed at the start
        yield ("arrive", bar("EPI"), 0)
        g0 = 0
        for it, n in enumerate(items):
            for gl in range((n + 1) // 2):
                g = g0 + gl
                yield ("wait", bar(("DQF", g & 1)), g >> 1)
                assert acc[q] == ("dq", g), f"drain({g}) reads {acc[q]}"
                acc[q] = ("read", g)
                yield ("arrive", bar(("DQE", g & 1)), g >> 1)
            yield ("wait", bar("ACC"), it)
            if by_kind:
                yield ("wait", bar("ACCB"), it)
            elif two_issuers and plant == "accb_prologue":
                yield ("wait", bar("ACCB"), it)
            elif two_issuers and it in odd_items:
                yield ("wait", bar("ACCB"), odd_items.index(it))
            assert counts.get((it, "dv"), 0) == n and counts.get((it, "dk"), 0) == n, \
                f"epilogue of item {it} reads {counts.get((it, 'dv'), 0)} dV, {counts.get((it, 'dk'), 0)} dK products"
            ready_for[q] = it + 1                             # read, then zeroed for the next item
            yield ("arrive", bar("EPI"), it + 1)
            g0 += (n + 1) // 2

    roles = [producer()]
    if by_kind:
        roles += [kind_issuer(0), kind_issuer(1)]
    else:
        roles += [main_issuer(0), main_issuer(1)] if two_issuers else [main_issuer(0)]
    roles += [softmax(g, q) for g in range(2) for q in range(4)]
    roles += [drain(q) for q in range(4)] + [dq_issuer()]
    schedule(roles, fifo, rnd, slow_role)


def schedule(roles, fifo, rnd, slow_role=None):
    """Runs coroutine roles and MMA FIFOs under a random schedule (see run)."""
    pending = {i: None for i in range(len(roles))}

    def advance(i):
        try:
            pending[i] = roles[i].send(None)
        except StopIteration:
            pending[i] = "done"

    for i in range(len(roles)):
        advance(i)
    steps = 0
    while True:
        steps += 1
        assert steps < 400000
        enabled = []
        for i, req in pending.items():
            if req == "done":
                continue
            if req[0] == "wait":
                _, br, k = req
                assert br.done <= k + 1, f"{br.name}: phase {k + 1} completed before a waiter for phase {k} passed"
                if br.passes(k):
                    enabled.append(("role", i))
            else:
                enabled.append(("role", i))
        for who, f in fifo.items():
            if f:
                enabled.append(("pipe", who))
        if not enabled:
            blocked = {i: (r[1].name, r[2], r[1].done) for i, r in pending.items() if r != "done"}
            assert not blocked, f"deadlock: {blocked}"
            return
        if slow_role is not None and len(enabled) > 1 and rnd.random() > 0.02:
            enabled = [e for e in enabled if e != ("role", slow_role)] or enabled
        kind, x = rnd.choice(enabled)
        if kind == "pipe":
            item = fifo[x].pop(0)
            if item[0] == "mma":
                item[1](item[2])
            else:
                item[1].arrive(item[2])
            continue
        req = pending[x]
        if req[0] == "wait":
            _, br, k = req
            assert br.done == k + 1, f"{br.name}: wait for phase {k} passed at {br.done} completed phases"
        elif req[0] == "arrive":
            req[1].arrive(req[2])
        advance(x)


def run_pair(nsub, NB, NST, seed, soft_waits_full, ordered=True):
    """One random schedule of a CTA pair in either pass of the two-pass mode.

    Per CTA r: a producer (stage s of sub-tile u, FULL_r(s) / EMPTY_r(s)) and
    two softmax warpgroups of four warps; in CTA 0 the two issuing threads:
    warp 10 issues S/dP(u) once the pair is ready (RDY, both producers) and,
    from u = NB on, once EMPTY(u-NB) shows the buffer's previous sub-tile
    consumed; warp 1 issues the PF(u)-gated product (dV/dK in pass 1, dQ in
    pass 2) and commits EMPTY(u).  Commits go to both CTAs' barriers (a
    multicast) and the softmax warps arrive on CTA 0's PF barrier (a remote
    arrive); both are modelled as deliveries that may land later.  Deliveries
    from one source (an issuing thread's commits, one warp's arrives) to one
    CTA land in the order they were made (a later commit tracks the earlier
    one's MMAs too); deliveries on different such channels interleave freely.
    soft_waits_full: pass 1's softmax also waits for its own stage.  ordered:
    False lets every delivery land in any order (see the test below)."""
    rnd = random.Random(seed)
    serial = [0]

    def channel(ch):
        serial[0] += 1
        return ch if ordered else (ch, serial[0])
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    for r in range(2):
        for b in range(NB):
            bar(("SF", r, b))
        for st in range(NST):
            bar(("FULL", r, st))
            bar(("EMPTY", r, st))
    for x in range(4):
        bar(("PF", x), 8)            # four warps of one warpgroup, in each CTA
    bar("RDY", 2)                    # both producers
    nready = min(nsub, NB)

    stage = {(r, st): None for r in range(2) for st in range(NST)}
    stage_use = {(r, st): set() for r in range(2) for st in range(NST)}
    tmem = {b: "free" for b in range(NB)}                        # the pair's buffer b, MMA side
    tq = {(r, b, q): None for r in range(2) for b in range(NB) for q in range(4)}
    fifo = {"w10": [], "w1": []}
    later = {}                                                    # (source, CTA) -> deliveries in flight

    def mma_sdp(u):
        b = u % NB
        assert tmem[b] == "free", f"S/dP({u}) overwrites buffer {b}"
        for r in range(2):
            assert stage[(r, u % NST)] == u, f"S/dP({u}) reads CTA {r}'s stage holding {stage[(r, u % NST)]}"
            stage_use[(r, u % NST)].add("sdp")
            for q in range(4):
                tq[(r, b, q)] = ("S", u)
        tmem[b] = ("S", u)

    def mma_second(u):
        b = u % NB
        for r in range(2):
            assert stage[(r, u % NST)] == u and "sdp" in stage_use[(r, u % NST)]
            stage_use[(r, u % NST)].add("second")
            for q in range(4):
                assert tq[(r, b, q)] == ("P", u), f"product({u}) reads {tq[(r, b, q)]}"
        tmem[b] = "free"

    def producer(r):
        for u in range(nsub):
            st = u % NST
            yield ("wait", bar(("EMPTY", r, st)), u // NST - 1)
            if stage[(r, st)] is not None:
                assert stage_use[(r, st)] >= {"sdp", "second"}, f"CTA {r} stage {st} reused early"
            stage[(r, st)] = u
            stage_use[(r, st)] = set()
            yield ("arrive", bar(("FULL", r, st)), u // NST)
            if u == nready - 1:
                for x in range(nready):
                    yield ("wait", bar(("FULL", r, x)), 0)
                yield ("arrive", bar("RDY"), 0)

    def warp10():
        yield ("wait", bar("RDY"), 0)
        for u in range(nsub):
            if u >= NB:
                w = u - NB
                yield ("wait", bar(("EMPTY", 0, w % NST)), w // NST)
            fifo["w10"].append(("mma", mma_sdp, u))
            fifo["w10"].append(("commit", [(("w10", r), bar(("SF", r, u % NB)), u // NB) for r in range(2)]))

    def warp1():
        for u in range(nsub):
            yield ("wait", bar(("PF", u % 4)), u // 4)
            fifo["w1"].append(("mma", mma_second, u))
            fifo["w1"].append(("commit", [(("w1", r), bar(("EMPTY", r, u % NST)), u // NST) for r in range(2)]))

    def softmax(r, grp, q):
        for u in range(grp, nsub, 2):
            b = u % NB
            yield ("wait", bar(("SF", r, b)), u // NB)
            if soft_waits_full:
                yield ("wait", bar(("FULL", r, u % NST)), u // NST)
            assert tq[(r, b, q)] == ("S", u), f"softmax({u}) reads {tq[(r, b, q)]}"
            tq[(r, b, q)] = ("P", u)
            if u + NB < nsub:
                v = u + NB
                yield ("wait", bar(("FULL", r, v % NST)), v // NST)
            yield ("remote", ("soft", r, grp, q), bar(("PF", u % 4)), u // 4)

    roles = [producer(0), producer(1), warp10(), warp1()]
    roles += [softmax(r, g, q) for r in range(2) for g in range(2) for q in range(4)]
    pending = {}

    def advance(i):
        try:
            pending[i] = roles[i].send(None)
        except StopIteration:
            pending[i] = "done"

    for i in range(len(roles)):
        advance(i)
    steps = 0
    while True:
        steps += 1
        assert steps < 400000
        enabled = []
        for i, req in pending.items():
            if req == "done":
                continue
            if req[0] == "wait":
                _, br, k = req
                assert br.done <= k + 1, f"{br.name}: phase {k + 1} completed before a waiter for phase {k} passed"
                if br.passes(k):
                    enabled.append(("role", i))
            else:
                enabled.append(("role", i))
        for who in fifo:
            if fifo[who]:
                enabled.append(("pipe", who))
        for ch, queue in later.items():
            if queue:
                enabled.append(("later", ch))
        if not enabled:
            blocked = {i: (r[1].name, r[2], r[1].done) for i, r in pending.items() if r != "done"}
            assert not blocked, f"deadlock: {blocked}"
            return
        kind, x = rnd.choice(enabled)
        if kind == "pipe":
            item = fifo[x].pop(0)
            if item[0] == "mma":
                item[1](item[2])
            else:
                for ch, br, k in item[1]:
                    later.setdefault(channel(ch), []).append((br, k))
            continue
        if kind == "later":
            br, k = later[x].pop(0)
            br.arrive(k)
            continue
        req = pending[x]
        if req[0] == "wait":
            _, br, k = req
            assert br.done == k + 1, f"{br.name}: wait for phase {k} passed at {br.done} completed phases"
        elif req[0] == "arrive":
            req[1].arrive(req[2])
        elif req[0] == "remote":
            later.setdefault(channel(req[1]), []).append((req[2], req[3]))
        advance(x)


@pytest.mark.parametrize("nsub", list(range(1, 12)) + [17, 26])
@pytest.mark.parametrize("NB,NST,soft_waits_full", [
    (3, 6, True), (2, 4, True),      # pass 1 (dK/dV), head_dim 32 and 64
    (3, 6, False), (2, 6, False),    # pass 2 (dQ), head_dim 32 and 64
])
def test_pair_protocol_random_schedules(nsub, NB, NST, soft_waits_full):
    """Both passes of the two-pass mode with their buffer and stage counts,
    25 random schedules each."""
    for seed in range(25):
        run_pair(nsub, NB, NST, seed * 7 + nsub, soft_waits_full)


def run_fwd(nk, seed, p_move, nsb=2, one_producer=False):
    """One random schedule of one forward CTA over nk key tiles: the producer
    (Q once; K tile j into stage j % 2 after KE, [V_lo | V_hi] tile j into
    stage j % 2 after VE; each copy lands on its own, in any order), the MMA
    issuer (S(0), S(1) after Q, K_0, K_1; then per tile: wait PF(j), P(j) V_j,
    commits VE and OD, S(j+2)) and four softmax warps (per tile: wait SF(j);
    with probability p_move the warp's row max moves, and for j > 0 it waits
    OD(j-1) and rescales its O rows; it writes P(j), waits for V_j and K_{j+2},
    arrives PF(j)).  K and V copies come from two independent producer lanes.
    nsb: the S buffers (2 at head_dim 64, 3 at head_dim <= 32):
    S(j) goes to buffer j % nsb after P(j - nsb) V, and the softmax waits for
    K_{j+nsb}.  one_producer: K_j and V_j issued in turn by one lane (the
    layout before K and V were split onto two lanes)."""
    rnd = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    nkst = nsb                                 # K stages, as many as S buffers
    for x in range(nkst):
        bar(("KF", x))
        bar(("KE", x))
    for x in range(2):
        bar(("VF", x))
        bar(("VE", x))
    for x in range(nsb):
        bar(("SF", x))
        bar(("PF", x), 4)
    bar(("OD", 0))
    bar(("OD", 1))                            # O updated after P(j) V_j, alternating by tile parity
    kst = {x: None for x in range(nkst)}
    kuse = {x: set() for x in range(nkst)}
    vst = {0: None, 1: None}
    vuse = {0: set(), 1: set()}
    sbuf = {b: "free" for b in range(nsb)}
    tq = {(b, q): None for b in range(nsb) for q in range(4)}
    o_last = {q: -1 for q in range(4)}        # last P V product applied to this warp's O rows
    o_pv = [-1]                               # last P V product executed
    fifo = []
    landing = []                              # copies in flight: (barrier, phase, effect)

    def mma_s(j):
        b = j % nsb
        assert sbuf[b] == "free", f"S({j}) overwrites buffer {b}"
        assert kst[j % nkst] == j, f"S({j}) reads K stage holding {kst[j % nkst]}"
        kuse[j % nkst].add("s")
        sbuf[b] = ("S", j)
        for q in range(4):
            tq[(b, q)] = ("S", j)

    def mma_pv(j):
        b = j % nsb
        for q in range(4):
            assert tq[(b, q)] == ("P", j), f"PV({j}) reads {tq[(b, q)]}"
            assert o_last[q] == j - 1, f"PV({j}) accumulates onto O rows holding PV({o_last[q]})"
            o_last[q] = j
        assert vst[j % 2] == j
        vuse[j % 2].add("pv")
        o_pv[0] = j
        sbuf[b] = "free"

    def producer_k():
        for j in range(nk):
            sk = j % nkst
            yield ("wait", bar(("KE", sk)), j // nkst - 1)
            if kst[sk] is not None:
                assert "s" in kuse[sk], f"K stage {sk} reused before S({kst[sk]}) read it"
            landing.append((bar(("KF", sk)), j // nkst, ("k", sk, j)))

    def producer_v():
        for j in range(nk):
            sv = j % 2
            yield ("wait", bar(("VE", sv)), j // 2 - 1)
            if vst[sv] is not None:
                assert "pv" in vuse[sv], f"V stage {sv} reused before PV({vst[sv]}) read it"
            landing.append((bar(("VF", sv)), j // 2, ("v", sv, j)))

    def issuer():
        for j in range(min(nsb, nk)):
            yield ("wait", bar(("KF", j % nkst)), j // nkst)
            fifo.append(("mma", mma_s, j))
            fifo.append(("commit", bar(("SF", j % nsb)), j // nsb))
            fifo.append(("commit", bar(("KE", j % nkst)), j // nkst))
        for j in range(nk):
            yield ("wait", bar(("PF", j % nsb)), j // nsb)
            fifo.append(("mma", mma_pv, j))
            fifo.append(("commit", bar(("VE", j % 2)), j // 2))
            fifo.append(("commit", bar(("OD", j & 1)), j >> 1))
            if j + nsb < nk:
                v = j + nsb
                fifo.append(("mma", mma_s, v))
                fifo.append(("commit", bar(("SF", v % nsb)), v // nsb))
                fifo.append(("commit", bar(("KE", v % nkst)), v // nkst))

    def softmax(q):
        for j in range(nk):
            b = j % nsb
            yield ("wait", bar(("SF", b)), j // nsb)
            assert tq[(b, q)] == ("S", j), f"softmax({j}) reads {tq[(b, q)]}"
            if j > 0 and rnd.random() < p_move:
                yield ("wait", bar(("OD", (j - 1) & 1)), (j - 1) >> 1)
                assert o_last[q] == j - 1, f"rescale at tile {j} sees O rows at PV({o_last[q]})"
            tq[(b, q)] = ("P", j)
            yield ("wait", bar(("VF", j % 2)), j // 2)
            if j + nsb < nk:
                yield ("wait", bar(("KF", (j + nsb) % nkst)), (j + nsb) // nkst)
            yield ("arrive", bar(("PF", j % nsb)), j // nsb)

    def producer_kv():
        # one lane: K_j, then V_j, for each j in turn
        for j in range(nk):
            sk, sv = j % nkst, j % 2
            yield ("wait", bar(("KE", sk)), j // nkst - 1)
            landing.append((bar(("KF", sk)), j // nkst, ("k", sk, j)))
            yield ("wait", bar(("VE", sv)), j // 2 - 1)
            landing.append((bar(("VF", sv)), j // 2, ("v", sv, j)))

    producers = [producer_kv()] if one_producer else [producer_k(), producer_v()]
    roles = producers + [issuer()] + [softmax(q) for q in range(4)]
    pending = {}

    def advance(i):
        try:
            pending[i] = roles[i].send(None)
        except StopIteration:
            pending[i] = "done"

    for i in range(len(roles)):
        advance(i)
    steps = 0
    while True:
        steps += 1
        assert steps < 200000
        enabled = []
        for i, req in pending.items():
            if req == "done":
                continue
            if req[0] == "wait":
                _, br, k = req
                assert br.done <= k + 1, f"{br.name}: phase {k + 1} completed before a waiter for phase {k} passed"
                if br.passes(k):
                    enabled.append(("role", i))
            else:
                enabled.append(("role", i))
        if fifo:
            enabled.append(("pipe", None))
        for x in range(len(landing)):
            enabled.append(("land", x))
        if not enabled:
            blocked = {i: (r[1].name, r[2], r[1].done) for i, r in pending.items() if r != "done"}
            assert not blocked, f"deadlock: {blocked}"
            return
        kind, x = rnd.choice(enabled)
        if kind == "pipe":
            item = fifo.pop(0)
            if item[0] == "mma":
                item[1](item[2])
            else:
                item[1].arrive(item[2])
            continue
        if kind == "land":
            br, k, (what, st, j) = landing.pop(x)
            if what == "k":
                kst[st], kuse[st] = j, set()
            else:
                vst[st], vuse[st] = j, set()
            br.arrive(k)
            continue
        req = pending[x]
        if req[0] == "wait":
            _, br, k = req
            assert br.done == k + 1, f"{br.name}: wait for phase {k} passed at {br.done} completed phases"
        elif req[0] == "arrive":
            req[1].arrive(req[2])
        advance(x)


@pytest.mark.parametrize("nk", list(range(1, 12)) + [25])
@pytest.mark.parametrize("p_move", [0.0, 0.3, 1.0])
def test_forward_protocol_random_schedules(nk, p_move):
    """The forward with row maxima that never move after the first tile, move
    sometimes, or move on every tile (each move waits for the previous P V
    product and rescales O), with two S buffers (head_dim 64) and three (head_dim
    <= 32); 30 random schedules each."""
    for seed in range(30):
        run_fwd(nk, seed * 31 + nk, p_move, nsb=2)
        run_fwd(nk, seed * 37 + nk, p_move, nsb=3)


@pytest.mark.parametrize("nk", [6, 9])
def test_forward_one_producer_lane_deadlocks_with_three_buffers(nk):
    """With K and V copies issued in turn by one lane and three S buffers, the
    lane waits for V stage (j % 2) to be freed by P(j-2) V, which needs the
    softmax of j-2 to see K_{j+1}, which the lane has not issued yet: every
    schedule deadlocks.  With two S buffers the softmax of j-2 waits for K_j,
    which the lane issued before V_j: no deadlock."""
    for seed in range(10):
        with pytest.raises(AssertionError, match="deadlock"):
            run_fwd(nk, seed, 0.3, nsb=3, one_producer=True)
        run_fwd(nk, seed, 0.3, nsb=2, one_producer=True)


def test_pair_protocol_relies_on_ordered_commits():
    """The pair kernels rely on one issuing thread's commits reaching a CTA in
    issue order: with every delivery free to land in any order, a softmax warp
    can find S/dP's barrier a phase behind and pass its parity test early."""
    failures = 0
    for seed in range(100):
        try:
            run_pair(7, 3, 6, seed, True, ordered=False)
        except AssertionError:
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("nsub", list(range(1, 12)) + [20])
def test_single_cta_dkdv_protocol_random_schedules(nsub):
    """The two-pass mode's single-CTA dK/dV pass (head_dim 16: 3 buffers, 6
    stages), 30 random schedules each."""
    for seed in range(30):
        run(nsub, False, 3, 6, seed * 13 + nsub, with_dq=False)


def run_dq_single(nsub, seed, NB=3, NST=4):
    """One random schedule of the two-pass mode's single-CTA dQ pass
    (tc_dq.cu): a producer (K/V stage s of key sub-tile v after EMPTY(s)), an
    MMA issuer (S/dP of the first NB sub-tiles after Q and their stages; per
    sub-tile: wait SD(v % NB), dQ += dS(v) K_v, commit EMPTY, S/dP(v+NB)) and
    four softmax warps that take every sub-tile (wait SF(v % NB), write dS over
    S, wait for the stage of v+NB, arrive SD(v % NB))."""
    rnd = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(name, count)
        return bars[name]

    for b in range(NB):
        bar(("SF", b))
        bar(("SD", b), 4)
    stage = {st: None for st in range(NST)}
    suse = {st: set() for st in range(NST)}
    tq = {(b, q): None for b in range(NB) for q in range(4)}
    tbuf = {b: "free" for b in range(NB)}
    fifo = []

    def mma_sdp(v):
        b = v % NB
        assert tbuf[b] == "free", f"S/dP({v}) overwrites buffer {b}"
        assert stage[v % NST] == v
        suse[v % NST].add("sdp")
        tbuf[b] = ("S", v)
        for q in range(4):
            tq[(b, q)] = ("S", v)

    def mma_dq(v):
        b = v % NB
        for q in range(4):
            assert tq[(b, q)] == ("dS", v), f"dQ({v}) reads {tq[(b, q)]}"
        assert stage[v % NST] == v and "sdp" in suse[v % NST]
        suse[v % NST].add("dq")
        tbuf[b] = "free"

    def producer():
        for v in range(nsub):
            st = v % NST
            yield ("wait", bar(("EMPTY", st)), v // NST - 1)
            if stage[st] is not None:
                assert suse[st] >= {"sdp", "dq"}, f"stage {st} reused early"
            stage[st], suse[st] = v, set()
            yield ("arrive", bar(("FULL", st)), v // NST)

    def issuer():
        for v in range(min(NB, nsub)):
            yield ("wait", bar(("FULL", v)), 0)
        for v in range(min(NB, nsub)):
            fifo.append(("mma", mma_sdp, v))
            fifo.append(("commit", bar(("SF", v % NB)), v // NB))
        for v in range(nsub):
            yield ("wait", bar(("SD", v % NB)), v // NB)
            fifo.append(("mma", mma_dq, v))
            fifo.append(("commit", bar(("EMPTY", v % NST)), v // NST))
            if v + NB < nsub:
                w = v + NB
                fifo.append(("mma", mma_sdp, w))
                fifo.append(("commit", bar(("SF", w % NB)), w // NB))

    def softmax(q):
        for v in range(nsub):
            b = v % NB
            yield ("wait", bar(("SF", b)), v // NB)
            assert tq[(b, q)] == ("S", v), f"softmax({v}) reads {tq[(b, q)]}"
            tq[(b, q)] = ("dS", v)
            if v + NB < nsub:
                w = v + NB
                yield ("wait", bar(("FULL", w % NST)), w // NST)
            yield ("arrive", bar(("SD", b)), v // NB)

    roles = [producer(), issuer()] + [softmax(q) for q in range(4)]
    pending = {}

    def advance(i):
        try:
            pending[i] = roles[i].send(None)
        except StopIteration:
            pending[i] = "done"

    for i in range(len(roles)):
        advance(i)
    while True:
        enabled = []
        for i, req in pending.items():
            if req == "done":
                continue
            if req[0] == "wait":
                _, br, k = req
                assert br.done <= k + 1, f"{br.name}: phase {k + 1} completed before a waiter for phase {k} passed"
                if br.passes(k):
                    enabled.append(i)
            else:
                enabled.append(i)
        if fifo:
            enabled.append("pipe")
        if not enabled:
            blocked = {i: (r[1].name, r[2], r[1].done) for i, r in pending.items() if r != "done"}
            assert not blocked, f"deadlock: {blocked}"
            return
        x = rnd.choice(enabled)
        if x == "pipe":
            item = fifo.pop(0)
            if item[0] == "mma":
                item[1](item[2])
            else:
                item[1].arrive(item[2])
            continue
        req = pending[x]
        if req[0] == "wait":
            assert req[1].done == req[2] + 1, f"{req[1].name}: wait for phase {req[2]} passed at {req[1].done}"
        elif req[0] == "arrive":
            req[1].arrive(req[2])
        advance(x)


@pytest.mark.parametrize("nsub", list(range(1, 12)) + [20])
def test_single_cta_dq_protocol_random_schedules(nsub):
    """The two-pass mode's single-CTA dQ pass (head_dim 16), 30 random
    schedules each."""
    for seed in range(30):
        run_dq_single(nsub, seed * 17 + nsub)


# (S/dP buffers, Q/dO stages, two main issuers): head_dim <= 32, head_dim 64,
# and the single-issuer form (head_dim 64 before its second issuer)
FUSED = [(3, 6, True), (2, 4, True), (2, 4, False)]


@pytest.mark.parametrize("nsub", list(range(1, 14)) + [20, 33])
@pytest.mark.parametrize("NB,NST,two", FUSED)
def test_fused_protocol_random_schedules(nsub, NB, NST, two):
    """The fused kernel: a dQ issuer, PF and SF rings of 8 and 2 NB; head_dim <=
    32 (two main issuers, one per sub-tile parity, 3 S/dP buffers, 6 Q/dO
    stages) and head_dim 64 (one main issuer, 2 buffers, 4 stages), odd and even
    sub-tile counts, 40 random schedules each."""
    for seed in range(40):
        run_fused(nsub, NB, NST, seed * 1000 + nsub, two)


@pytest.mark.parametrize("slow", [1, 2])
def test_fused_two_issuers_need_the_longer_ring(slow):
    """With two main issuers a PF ring of 4 is not enough: the issuer of one
    parity can fall behind until a later phase of its PF barrier completes
    before it saw the earlier one.  The model finds such schedules when that
    issuer (role 1 or 2) runs slowly; with the kernel's ring of 8 it finds none."""
    failures = 0
    for seed in range(200):
        try:
            run_fused(20, 3, 6, seed, True, pf_ring=4, slow_role=slow)
        except AssertionError:
            failures += 1
    assert failures > 0
    for seed in range(200):
        run_fused(20, 3, 6, seed, True, slow_role=slow)


def test_single_drain_barrier_aliases():
    """Why the drain barrier alternates: with a single barrier, at head_dim 64
    with an odd sub-tile count the softmax of the last (even) sub-tile waits for
    the drain of group g-1 while the drain of group g-2 may still be open, so
    its parity test can pass a phase early (and the dQ product of group g could
    overwrite group g-1's accumulator before it was read)."""
    failures = 0
    for seed in range(200):
        try:
            run(5, False, 2, 4, seed, dqe_pair=False)
        except AssertionError:
            failures += 1
    assert failures > 0


def test_model_catches_a_broken_protocol():
    """The fused model is not vacuous: without the softmax's wait for the dQ
    product, some schedule overwrites a dS block that dQ has not read; with the
    S^T product issued before dV (which reads the same half), some schedule
    overwrites P before dV read it."""
    for plant, msg in (("no_dqf_wait", "before its dQ product read it"), ("s_before_dv", "overwrites")):
        failures = 0
        for seed in range(200):
            try:
                run_fused(12, 3, 6, seed, True, plant=plant)
            except AssertionError as e:
                assert msg in str(e), (plant, str(e))
                failures += 1
        assert failures > 0, plant


@pytest.mark.parametrize("NB,NST,two", FUSED)
def test_fused_protocol_with_one_slow_role(NB, NST, two):
    """The fused kernel's protocol with each role in turn running slowly (the
    producer, either main issuer, a softmax warp, a drain warp, the dQ issuer):
    skewed schedules reach interleavings that uniform ones rarely do."""
    nroles = 1 + (2 if two else 1) + 8 + 4 + 1
    slows = list(range(nroles)) + ["main", "dq"] + (["main1"] if two else [])
    for slow in slows:
        for seed in range(12):
            run_fused(17, NB, NST, seed * 31 + len(str(slow)), two, slow_role=slow)




PERSISTENT_ITEMS = [[7, 7, 7], [7, 7, 7, 7, 7, 7, 7], [4, 4, 4, 3, 1], [1, 1, 1, 1], [2, 3, 2, 5], [25, 25],
                    [3, 6, 9], [1, 2, 1, 2, 6], [5, 1, 4]]


# (NB, NST, two issuers, K/V buffers, dK reads dS from the shared ring, dK
# before dP(u+NB), the ring guarded by QE(u-4) instead of DSE barriers, a
# P-ready barrier): head_dim <= 32 (two K/V tiles, the next item's loaded
# while the current one runs; dS from the ring), head_dim 64 (one K/V tile,
# dS from TMEM, P-ready), and variants
PERSIST = [(3, 6, True, 2, True, True, True, False), (2, 4, True, 1, False, False, False, True),
           (2, 4, True, 1, False, False, False, False), (3, 6, True, 1, False, False, False, False),
           (2, 4, False, 1, False, False, False, False), (2, 4, True, 2, True, False, False, False),
           (2, 4, True, 1, True, True, False, False), (3, 6, True, 2, True, True, False, False),
           (2, 4, True, 1, True, True, True, False), (3, 6, True, 2, True, True, True, True)]
PERSIST_NAMES = "NB,NST,two,kvbuf,ds_smem,dk_first,dse_by_qe,p_ready"


@pytest.mark.parametrize("items", PERSISTENT_ITEMS + [[1, 1, 1, 1, 1, 1], [1, 2, 1, 1, 3, 1]],
                         ids=lambda x: "-".join(map(str, x)))
@pytest.mark.parametrize(PERSIST_NAMES, PERSIST)
def test_persistent_protocol_random_schedules(items, NB, NST, two, kvbuf, ds_smem, dk_first, dse_by_qe, p_ready):
    """The persistent fused kernel over several work items per CTA (whole units
    of 7 or 25 sub-tiles as at N = 400 and N = 1600, split pieces, single
    sub-tiles, mixed parities, runs of one-sub-tile items), both head_dim
    variants, 25 random schedules each."""
    for seed in range(25):
        run_persistent(items, NB, NST, seed * 7919 + sum(items), two, kvbuf=kvbuf, ds_smem=ds_smem,
                       dk_first=dk_first, dse_by_qe=dse_by_qe, p_ready=p_ready)


@pytest.mark.parametrize(PERSIST_NAMES, PERSIST)
def test_persistent_protocol_with_one_slow_role(NB, NST, two, kvbuf, ds_smem, dk_first, dse_by_qe, p_ready):
    """Each role of the persistent CTA in turn running slowly, over items of odd
    and even lengths."""
    nroles = 1 + (2 if two else 1) + 8 + 4 + 1
    slows = list(range(nroles)) + ["main", "dq"] + (["main1"] if two else [])
    kw = dict(kvbuf=kvbuf, ds_smem=ds_smem, dk_first=dk_first, dse_by_qe=dse_by_qe, p_ready=p_ready)
    for slow in slows:
        for seed in range(8):
            run_persistent([3, 7, 2, 5], NB, NST, seed * 131 + len(str(slow)), two, slow_role=slow, **kw)
            run_persistent([1, 2, 1, 4], NB, NST, seed * 137 + len(str(slow)), two, slow_role=slow, **kw)


def test_persistent_model_catches_missing_item_waits():
    """The persistent model is not vacuous: without the issuers' wait for the
    previous item's epilogue, some schedule zeroes the accumulators before the
    epilogue read them; without the K/V producer's wait for KVE, some schedule
    loads the next item's K/V while the current item still reads its tile (with
    two K/V buffers: the item after next, while a slow dQ issuer still reads
    the tile of the item two before); without the softmax's DSE wait (or, in
    the form without DSE barriers, its wait for QE of sub-tile u-4), some
    schedule writes a dS ring block before the dK product of its previous
    sub-tile has read it."""
    # roles: the producer, 2 issuers, 8 softmax warps, then the drain warps
    for plant, msg, slow, kvbuf, items, by_qe in (
            ("no_epi_wait", "adds to accumulators", 11, 1, [3, 4, 3, 2], False),
            ("no_kve_wait", "still reads its tile", None, 1, [3, 4, 3, 2], False),
            ("no_kve_wait", "still reads its tile", "dq", 2, [3, 4, 3, 2], False),
            ("no_dse_wait", "['dk'] product read it", "main1", 2, [3, 4, 3, 2, 5], False),
            ("no_dse_wait", "['dk'] product read it", "main1", 2, [3, 4, 3, 2, 5], True)):
        failures = 0
        for seed in range(300):
            try:
                run_persistent(items, 3, 6, seed, True, plant=plant, slow_role=slow, kvbuf=kvbuf,
                               ds_smem=plant == "no_dse_wait", dk_first=plant == "no_dse_wait", dse_by_qe=by_qe)
            except AssertionError as e:
                assert msg in str(e), (plant, str(e))
                failures += 1
        assert failures > 0, plant


def test_persistent_prologue_waits_that_alias():
    """Why the odd issuer commits ACCB only for items it has a sub-tile in, and
    the prologue waits for its latest ACCB phase: (1) with an ACCB commit every
    item, an issuer without a sub-tile in an item commits after the previous
    epilogue alone, and ACCB can complete two phases before the prologue issuer
    looks at it; (2) waiting instead for the odd issuer's last QE commit of the
    previous item lets the prologue issuer, with 4 stages and 2 buffers (head_dim
    64), find that stage barrier two phases behind when the odd issuer is slow."""
    for plant, items, NB, NST, slow in (("accb_prologue", [2, 1, 1, 1, 2, 1], 3, 6, "main"),
                                        ("qe_prologue", [4, 8, 5, 4, 2], 2, 4, 2)):
        failures = 0
        for seed in range(300):
            try:
                run_persistent(items, NB, NST, seed, True, plant=plant, slow_role=slow)
            except AssertionError as e:
                assert "completed before a waiter" in str(e) or "passed at" in str(e), str(e)
                failures += 1
        assert failures > 0, plant


def test_p_ready_model_catches_missing_waits():
    """The P-ready form (head_dim 64) is not vacuous: an issuer that issues
    dK(u) and dP(u+NB) without waiting for PF(u), or a softmax that arrives
    PR(u) before the stage of u+NB is loaded, fails in some schedule."""
    for plant, msgs in (("no_pf_after_pr", ("reads dS", "reads ('dP'")), ("pr_without_stage", ("reads stage",))):
        failures = 0
        for slow in (None, 2, 6, "main"):
            for seed in range(60):
                try:
                    run_persistent([5, 7, 4], 2, 4, seed, True, slow_role=slow, plant=plant, p_ready=True)
                except AssertionError as e:
                    assert any(m in str(e) for m in msgs), (plant, str(e))
                    failures += 1
        assert failures > 0, plant



def test_lagged_issue_form():
    """The lagged issue form (one issuer wait per sub-tile: dK / dP of the
    previous sub-tile issued after the next PR) is sound with 6 stages and 3
    S/dP buffers (head_dim <= 32) and deadlocks with 4 stages and 2 buffers
    (head_dim 64): the stage that S(u+NB) needs is freed only by a dK that
    waits for that S's softmax."""
    kw = dict(kvbuf=2, ds_smem=True, dk_first=True, dse_by_qe=True, p_ready=True, lag=True)
    for items in ([9, 5, 6], [3, 7, 2, 5], [1, 2, 1, 4]):
        for seed in range(20):
            run_persistent(items, 3, 6, seed, True, **kw)
    deadlocks = 0
    for seed in range(20):
        try:
            run_persistent([7, 7], 2, 4, seed, True, kvbuf=1, p_ready=True, lag=True)
        except AssertionError as e:
            assert "deadlock" in str(e), str(e)
            deadlocks += 1
    assert deadlocks > 0


def test_issuers_by_kind_form():
    """The issuers split by MMA kind (one takes dV and S after PR, the other dK
    and dP after PF; a stage freed by both) is sound at both head_dim
    variants under random and slow-role schedules, and still needs its EPI
    and stage waits."""
    for NB, NST, kw in ((3, 6, dict(kvbuf=2, ds_smem=True, dk_first=True, dse_by_qe=True)), (2, 4, dict(kvbuf=1))):
        for items in ([9, 5, 6], [3, 7, 2, 5], [1, 2, 1, 4], [1, 1, 1]):
            for seed in range(10):
                run_persistent(items, NB, NST, seed, True, p_ready=True, by_kind=True, **kw)
                run_persistent(items, NB, NST, seed, True, p_ready=True, by_kind=True, slow_role="main1", **kw)
        for plant in ("no_epi_wait", "pr_without_stage"):
            failures = 0
            for slow in (None, 2, 11, "main"):
                for seed in range(30):
                    try:
                        run_persistent([5, 7, 4, 3], NB, NST, seed, True, slow_role=slow, plant=plant, p_ready=True,
                                       by_kind=True, **kw)
                    except AssertionError:
                        failures += 1
            assert failures > 0, (NB, plant)
