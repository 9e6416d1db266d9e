"""A randomised model of the tensor-core decode's barrier protocol.

One unit of the kernel runs on a cluster of a score CTA (0) and a value CTA
(1).  Their warps hand tiles to each other through mbarriers (phase counting
with parity waits), bulk copies that complete transaction bytes, and
tensor-core commits that arrive when the issuing thread's MMAs are done.
This module re-states that protocol as it is written in
`mla_decode_context_gb300/csrc/dcp_decode_tc.cu` (the same barriers, counts,
parities and ring sizes, role by role) and runs it under random
interleavings, with every asynchronous completion (copies landing, MMAs
finishing, remote arrivals) delivered at a random later time.

Two forms of the protocol, as the kernel has them:
  * bf16 cache (``decoupled=True``): each CTA loads what it needs: the score
    CTA the whole tile into its stage, the value CTA chunks 4-7 into its own
    ring and (group 2) chunks 0-3 into its receive ring.  Only P crosses the
    cluster, and a stage is free once S is done;
  * fp8 cache (``decoupled=False``): the score CTA loads chunks 0-3 and 8,
    the value CTA chunks 4-7, and each copies the 16 KB its peer lacks: the
    value CTA's forwarder into the score CTA's stage, the score CTA's
    forwarder into the value CTA's receive ring.

What a run checks:
  * no deadlock, and no arrival beyond a barrier's count;
  * no phase completed by arrivals meant for different tiles (each arrival
    names its tile; an early arrival for a later tile that lands in an
    earlier tile's open phase would let that phase complete too soon);
  * no aliased wait: a parity wait never passes while its barrier is a phase
    behind the one it targets (the parity of phase t - 1 equals that of
    t + 1), nor is a wait left behind by two phases;
  * no buffer is overwritten while a reader still needs its previous
    contents, and no reader starts before its data is complete: the stage
    ring, the value CTA's own and receive rings, the P slots and their
    staging, the S slots, the running-max ring and the row-mask ring.

It is test infrastructure: the kernel does not use it.
"""
from __future__ import annotations

import random

# ring sizes and counts as in the kernel
K_STAGES, K_OWN, K_RECV, K_SBUF, K_SPARTS, K_PSLOTS = 5, 7, 4, 2, 3, 4
HALF = 16384            # bytes forwarded each way per tile (four 4 KB chunks)
PTX = 128 * 32 * 2 + 128 * 4   # bytes that fill one P slot


class ProtocolError(AssertionError):
    pass


class Bar:
    """An mbarrier: `count` arrivals and a transaction count per phase."""

    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending, self.tx, self.done = count, 0, 0
        self.tag = None         # the tile the open phase's arrivals are for

    def arrive(self, n=1, tag=None):
        if tag is not None:
            if self.tag is None:
                self.tag = tag
            elif self.tag != tag:
                raise ProtocolError("%s: phase %d mixes arrivals for tiles %s and %s"
                                    % (self.name, self.done, self.tag, tag))
        self.pending -= n
        if self.pending < 0:
            raise ProtocolError("over-arrival on %s (phase %d)" % (self.name, self.done))
        self._check()

    def txop(self, b):
        self.tx += b
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count
            self.tag = None


class Model:
    def __init__(self, ntiles, seed, rescale_prob=0.3, mutation=None, decoupled=True):
        # `mutation` plants one mistake in the protocol (for the tests that
        # show the checks catch it): see MUTATIONS
        self.mut = mutation
        self.decoupled = decoupled
        self.n = ntiles
        self.rng = random.Random(seed)
        self.rescale_prob = rescale_prob
        self.bars = {}
        self.delayed = []          # (ready time, callable or ("fifo", key))
        self.clock = 0
        self.fifo = {}             # per issuing thread: ordered completions
        self._mk_barriers()
        # buffer state: what each buffer holds and who still needs it
        self.stage = [dict(tile=None, own=False, fwd=False, s_done=set(), cp_read=True)
                      for _ in range(K_STAGES)]
        self.own = [dict(tile=None, landed=False, fwd_read=True, pv_read=True, fenced=False) for _ in range(K_OWN)]
        self.recv = [dict(tile=None, landed=False, pv_read=True, fenced=False) for _ in range(K_RECV)]
        self.pslot = [dict(tile=None, bytes=0, pv_read=True, max_read=True) for _ in range(K_PSLOTS)]
        self.stg = [dict(tile=None, reads_left=0) for _ in range(K_PSLOTS)]
        self.sslot = [dict(tile=None, parts_done=0, read=True) for _ in range(K_SBUF)]
        self.mring = [dict(tile=None, reads_left=0) for _ in range(8)]
        self.mask = [dict(tile=None, read=True) for _ in range(16)]
        self.pv_done_tiles = set()
        self.claimed = [0, 0]

    # ---------------------------------------------------------------- set-up
    def _mk_barriers(self):
        def mk(cta, name, n, count):
            for i in range(n):
                self.bars[(cta, name, i)] = Bar("%s[%d]@%d" % (name, i, cta), count)
        for cta in (0, 1):
            mk(cta, "kv_loaded", K_STAGES, 128)
            mk(cta, "kv_full", K_STAGES, 4 if self.mut == "kv_full_without_fence" else 5)
            mk(cta, "s_done", K_STAGES, K_SPARTS if self.decoupled else K_SPARTS + 1)
            mk(cta, "own_loaded", K_OWN, 128)
            mk(cta, "own_free", K_OWN, 1)
            mk(cta, "v_full", K_RECV, 128 if self.decoupled else 1)
            mk(cta, "v_free", K_RECV, 1)
            mk(cta, "s_full", K_SBUF, K_SPARTS + 1)
            mk(cta, "s_free", K_SBUF, 4)
            mk(cta, "q_ready", 1, 8)
            mk(cta, "q_gone", 1, 1)
            mk(cta, "p_full", K_PSLOTS, 1)
            mk(cta, "p_free", K_PSLOTS, 1)
            mk(cta, "p_ok", K_PSLOTS, 5)
            mk(cta, "pv_done", K_PSLOTS, 1)
            mk(cta, "o_final", 1, 1)
            mk(cta, "fin_l", 1, 1)
            mk(cta, "m_pub", 8, 4)
            mk(cta, "sm_fin", 1, 8)
        # value CTA arming at set-up
        for i in range(K_PSLOTS):
            self.b(1, "p_full", i).txop(PTX)
            self.b(1, "p_full", i).arrive()
        if not self.decoupled:
            for i in range(K_RECV):
                self.b(1, "v_full", i).txop(HALF)
                self.b(1, "v_full", i).arrive()
        self.b(1, "fin_l", 0).txop(128 * 4)
        self.b(1, "fin_l", 0).arrive()

    def b(self, cta, name, i):
        return self.bars[(cta, name, i)]

    # --------------------------------------------------------------- helpers
    def claim_stage(self, st, j, who):
        s = self.stage[st]
        if s["tile"] is not None:
            self.check(len(s["s_done"]) == K_SPARTS,
                       "%s overwrote stage %s (tile %s) before S(%s) finished", who, st, j, s["tile"])
            self.check(s["cp_read"], "%s overwrote stage %s (tile %s) before tile %s's chunks 0-3 were copied", who, st, j, s["tile"])
        self.stage[st] = dict(tile=j, own=False, fwd=False, s_done=set(), cp_read=self.decoupled)

    def _delay(self):
        # heavy-tailed: most completions are quick, a few take very long
        return int(self.rng.paretovariate(1.1) * 2)

    def later(self, fn, fifo=None):
        """An asynchronous completion, delivered at a random later time (in
        issue order among those of one issuing thread)."""
        if fifo is None:
            self.delayed.append((self.clock + self._delay(), fn))
        else:
            q = self.fifo.setdefault(fifo, [])
            q.append(fn)
            if len(q) == 1:
                self.delayed.append((self.clock + self._delay(), ("fifo", fifo)))

    def _deliver(self, item):
        if isinstance(item, tuple) and item[0] == "fifo":
            q = self.fifo[item[1]]
            fn = q.pop(0)
            fn()
            if q:
                self.delayed.append((self.clock + self._delay(), ("fifo", item[1])))
        else:
            item()

    @staticmethod
    def W(cta, name, i, t):
        """Wait for phase t of a barrier (parity wait)."""
        return ("wait", cta, name, i, t)

    def check(self, cond, fmt, *args):
        if not cond:
            raise ProtocolError(fmt % args)

    # ----------------------------------------------------------------- roles
    def q_load(self):
        # warps 0-7 of the score CTA move Q to TMEM and arrive on q_ready
        for _ in range(8):
            yield ("do", lambda: self.b(0, "q_ready", 0).arrive())

    def score_producers(self, g):
        yield self.W(0, "q_ready", 0, 0)
        for j in range(g, self.n, 2):
            st = j % K_STAGES
            if j >= 5 and self.mut != "producers_uncoupled":
                # the other group has claimed its stage for tile j - 5 (a
                # monotonic count, so no parity to alias)
                need = ((j - 5) >> 1) + 1
                yield ("cond", lambda need=need, g=g: self.claimed[1 - g] >= need)
            if self.mut != "producers_skip_stage_free":
                yield self.W(0, "s_done", st, j // K_STAGES - 1)

            def claim(j=j, g=g):
                self.claimed[g] = max(self.claimed[g], (j >> 1) + 1)
            yield ("do", claim)

            def write(j=j, st=st):
                s = self.stage[st]
                if s["tile"] == j:      # the value CTA's half landed first and claimed it
                    s["own"] = False
                else:
                    self.claim_stage(st, j, "score producers")
                m = self.mask[j % 16]
                self.check(m["read"], "mask slot %s overwritten before tile %s's softmax", j % 16, m["tile"])
                self.mask[j % 16] = dict(tile=j, read=False)
            yield ("do", write)
            # fp8: warp 0 arms the value CTA's 16 KB; the other warps arrive
            if self.decoupled:
                yield ("do", lambda st=st, j=j: self.b(0, "kv_full", st).arrive(tag=j))
            else:
                yield ("do", lambda st=st, j=j: (self.b(0, "kv_full", st).txop(HALF),
                                                  self.b(0, "kv_full", st).arrive(tag=j)))
            for _ in range(3):
                yield ("do", lambda st=st, j=j: self.b(0, "kv_full", st).arrive(tag=j))

            def landed(j=j, st=st):
                self.stage[st]["own"] = True
                if self.decoupled:      # bf16: the whole tile is this CTA's own load
                    self.stage[st]["fwd"] = True
                self.b(0, "kv_loaded", st).arrive(128)
            yield ("do", lambda f=landed: self.later(f))

    def value_producers(self, g):
        for j in range(g, self.n, 2):
            os_ = j % K_OWN
            yield self.W(1, "own_free", os_, j // K_OWN - 1)

            def write(j=j, os_=os_):
                o = self.own[os_]
                self.check(o["fwd_read"] and o["pv_read"],
                           "own slot %s overwritten (tile %s) while tile %s still needed", os_, j, o["tile"])
                self.own[os_] = dict(tile=j, landed=False, fwd_read=self.decoupled, pv_read=False, fenced=False)
            yield ("do", write)

            def landed(j=j, os_=os_):
                self.own[os_]["landed"] = True
                self.b(1, "own_loaded", os_).arrive(128)
            yield ("do", lambda f=landed: self.later(f))

    def value_recv_producers(self):
        """bf16: the value CTA's group 2 loads chunks 0-3 of every tile into
        receive slot j % K_RECV once PV(j - K_RECV) has freed it."""
        for j in range(self.n):
            vs = j % K_RECV
            if self.mut != "recv_producers_skip_slot_free":
                yield self.W(1, "v_free", vs, j // K_RECV - 1)

            def write(j=j, vs=vs):
                r = self.recv[vs]
                self.check(r["pv_read"], "receive slot %s overwritten (tile %s) before PV(%s)", vs, j, r["tile"])
                self.recv[vs] = dict(tile=j, landed=False, pv_read=False, fenced=False)
            yield ("do", write)

            def landed(j=j, vs=vs):
                self.recv[vs]["landed"] = True
                self.b(1, "v_full", vs).arrive(128)
            yield ("do", lambda f=landed: self.later(f))

    def score_forwarder(self):
        yield self.W(0, "q_ready", 0, 0)
        if not self.decoupled:
            yield ("do", lambda: self.later(lambda: self.b(1, "q_gone", 0).arrive()))
        jf = jc = 0
        while jc < self.n:
            moved = False
            if jf < self.n and self.passed(0, "kv_loaded", jf % K_STAGES, jf // K_STAGES, "score fwd"):
                st = jf % K_STAGES
                self.check(self.stage[st]["tile"] == jf and self.stage[st]["own"],
                           "forwarder fenced stage %s for tile %s before its rows landed", st, jf)
                if self.mut != "kv_full_without_fence":
                    yield ("do", lambda st=st, jf=jf: self.b(0, "kv_full", st).arrive(tag=jf))
                jf += 1
                moved = True
            if self.decoupled:
                jc = jf     # bf16: no copies; the forwarder only fences
            elif jc < jf and self.passed(0, "v_free", jc % K_RECV, jc // K_RECV - 1, "score fwd"):
                st, rs, j = jc % K_STAGES, jc % K_RECV, jc

                def copy(st=st, rs=rs, j=j):
                    r = self.recv[rs]
                    self.check(r["pv_read"], "receive slot %s overwritten (tile %s) before PV(%s)", rs, j, r["tile"])
                    self.check(self.stage[st]["tile"] == j, "copy of tile %s from a stage holding %s", j, self.stage[st]["tile"])
                    self.recv[rs] = dict(tile=j, landed=False, pv_read=False, fenced=True)

                    def land():
                        self.stage[st]["cp_read"] = True
                        self.recv[rs]["landed"] = True
                        self.b(1, "v_full", rs).txop(-HALF)
                    self.later(land)
                yield ("do", copy)
                jc += 1
                moved = True
            if not moved:
                yield ("yield",)

    def value_forwarder(self):
        yield self.W(1, "q_gone", 0, 0)
        for j in range(self.n):
            st, os_ = j % K_STAGES, j % K_OWN
            yield self.W(1, "own_loaded", os_, j // K_OWN)
            yield self.W(1, "s_done", st, j // K_STAGES - 1)

            def copy(j=j, st=st, os_=os_):
                o = self.own[os_]
                self.check(o["tile"] == j and o["landed"], "value forwarder copies own slot %s before tile %s landed", os_, j)

                def land():
                    o["fwd_read"] = True
                    # the score producers may not have claimed the stage for j yet
                    if self.stage[st]["tile"] != j:
                        self.claim_stage(st, j, "the value CTA's copy")
                    self.stage[st]["fwd"] = True
                    self.b(0, "kv_full", st).txop(-HALF)
                self.later(land)
            yield ("do", copy)

    def recv_warp(self):
        for j in range(self.n):
            st, vs, os_ = j % K_STAGES, j % K_RECV, j % K_OWN
            if not (self.decoupled and self.mut == "recv_skips_v_full"):
                yield self.W(1, "v_full", vs, j // K_RECV)

            def arrivals(st=st, vs=vs, j=j):
                self.b(1, "v_full", vs).txop(HALF)
                self.b(1, "v_full", vs).arrive()
                self.b(1, "s_done", st).arrive(tag=j)
                self.later(lambda: self.b(0, "s_done", st).arrive(tag=j))
            if not self.decoupled:
                yield ("do", arrivals)
            if self.mut != "recv_skips_own_rows":
                yield self.W(1, "own_loaded", os_, j // K_OWN)

            def fence(j=j, os_=os_, vs=vs):
                # the proxy fence that makes the own slot's copies (and, bf16,
                # the receive slot's) visible to PV
                o = self.own[os_]
                if o["tile"] == j and o["landed"]:
                    o["fenced"] = True
                r = self.recv[vs]
                if self.decoupled and r["tile"] == j and r["landed"]:
                    r["fenced"] = True
            yield ("do", fence)
            yield ("do", lambda slot=j % K_PSLOTS, j=j: self.b(1, "p_ok", slot).arrive(tag=j))

    def s_issuer(self, b, part):
        yield self.W(0, "q_ready", 0, 0)
        for j in range(b, self.n, K_SBUF):
            st, u = j % K_STAGES, j // K_SBUF
            if self.mut != "issuers_skip_s_free":
                yield self.W(0, "s_free", b, u - 1)
            yield self.W(0, "kv_full", st, j // K_STAGES)

            def issue(j=j, st=st):
                s = self.stage[st]
                self.check(s["tile"] == j and s["own"] and s["fwd"],
                           "S(%s) part %s issued on stage %s holding tile %s (own %s, fwd %s)", j, part, st, s["tile"], s["own"], s["fwd"])
                sl = self.sslot[b]
                if sl["tile"] != j:   # the first part of S(j) to issue claims the slot
                    self.check(sl["read"], "S slot %s rewritten (tile %s) before the softmax read tile %s",
                               b, j, sl["tile"])
                    self.sslot[b] = dict(tile=j, parts_done=0, read=False)
                if part == 0:
                    self.b(0, "s_full", b).arrive(tag=j)

                def done():
                    sl2 = self.sslot[b]
                    self.check(sl2["tile"] == j, "S(%s) part %s completed into slot %s holding %s",
                               j, part, b, sl2["tile"])
                    sl2["parts_done"] += 1
                    self.stage[st]["s_done"].add(part)
                    self.b(0, "s_full", b).arrive(tag=j)
                    self.b(0, "s_done", st).arrive(tag=j)
                    self.b(1, "s_done", st).arrive(tag=j)
                self.later(done, fifo=("S", b, part))
            yield ("do", issue)

    def softmax(self, g):
        for j in range(g, self.n, 2):
            b, slot = j % K_SBUF, j % K_PSLOTS
            k = 0 if j == 1 else j - 3
            if k >= 0 and self.mut != "softmax_skips_m_pub":
                yield self.W(0, "m_pub", k % 8, k // 8)

                def read_m(k=k, j=j):
                    m = self.mring[k % 8]
                    self.check(m["tile"] == k, "tile %s read tile %s's max from ring slot %s, wanted %s", j, m["tile"], k % 8, k)
                    m["reads_left"] -= 1
                yield ("do", read_m)
            yield self.W(0, "s_full", b, j // K_SBUF)

            def read_s(j=j, b=b):
                sl = self.sslot[b]
                self.check(sl["tile"] == j and sl["parts_done"] == K_SPARTS,
                           "softmax read S slot %s for tile %s: holds %s with %s parts done", b, j, sl["tile"], sl["parts_done"])
                m = self.mask[j % 16]
                self.check(m["tile"] == j, "mask slot %s holds tile %s, wanted %s", j % 16, m["tile"], j)
                m["read"] = True
                sl["read"] = True
            yield ("do", read_s)
            for _ in range(4):
                yield ("do", lambda b=b, j=j: self.b(0, "s_free", b).arrive(tag=j))

            def post(j=j):
                m = self.mring[j % 8]
                self.check(m["reads_left"] <= 0, "max ring slot %s rewritten (tile %s) with tile %s unread", j % 8, j, m["tile"])
                # read by tile j + 3, and tile 0's also by tile 1
                readers = [r for r in (j + 3, 1 if j == 0 else None) if r is not None and r < self.n]
                self.mring[j % 8] = dict(tile=j, reads_left=len(readers))
            yield ("do", post)
            for _ in range(4):
                yield ("do", lambda j=j: self.b(0, "m_pub", j % 8).arrive(tag=j))
            if self.mut != "softmax_skips_p_free":
                yield self.W(0, "p_free", slot, j // K_PSLOTS - 1)

            def send(j=j, slot=slot):
                s = self.stg[slot]
                self.check(s["reads_left"] == 0, "P staging slot %s rewritten (tile %s) before its copies read it", slot, j)
                p = self.pslot[slot]
                self.check(p["pv_read"] and p["max_read"],
                           "P slot %s refilled (tile %s) before tile %s was consumed", slot, j, p["tile"])
                self.stg[slot] = dict(tile=j, reads_left=8)
                self.pslot[slot] = dict(tile=j, bytes=0, pv_read=False, max_read=False)
                for _ in range(8):      # two bulk copies per warp
                    def land(slot=slot):
                        self.stg[slot]["reads_left"] -= 1
                        self.pslot[slot]["bytes"] += PTX // 8
                        self.b(1, "p_full", slot).txop(-(PTX // 8))
                    self.later(land)
            yield ("do", send)
        for _ in range(4):
            yield ("do", lambda: self.b(0, "sm_fin", 0).arrive())
        if g == 0:
            yield self.W(0, "sm_fin", 0, 0)
            yield ("do", lambda: self.later(lambda: self.b(1, "fin_l", 0).txop(-(128 * 4))))

    def value_max(self):
        m_prev_set = False
        for j in range(self.n):
            slot = j % K_PSLOTS
            yield self.W(1, "p_full", slot, j // K_PSLOTS)

            def rearm(slot=slot, j=j):
                p = self.pslot[slot]
                self.check(p["tile"] == j and p["bytes"] == PTX, "P(%s) seen incomplete in slot %s", j, slot)
                p["max_read"] = True
                self.b(1, "p_full", slot).txop(PTX)
                self.b(1, "p_full", slot).arrive()
            yield ("do", rearm)
            if m_prev_set and self.rng.random() < self.rescale_prob:
                jp = j - 1
                yield self.W(1, "pv_done", jp % K_PSLOTS, jp // K_PSLOTS)
                yield ("do", lambda jp=jp: self.check(jp in self.pv_done_tiles,
                                                      "O rescaled before PV(%s) finished", jp))
            m_prev_set = True
            for _ in range(4):
                yield ("do", lambda slot=slot, j=j: self.b(1, "p_ok", slot).arrive(tag=j))

    def pv_issuer(self):
        for j in range(self.n):
            vs, os_, slot = j % K_RECV, j % K_OWN, j % K_PSLOTS
            yield self.W(1, "p_ok", slot, j // K_PSLOTS)

            def issue(j=j, vs=vs, os_=os_, slot=slot):
                self.check(self.pslot[slot]["tile"] == j and self.pslot[slot]["bytes"] == PTX,
                           "PV(%s) issued before P landed", j)
                self.check(self.recv[vs]["tile"] == j and self.recv[vs]["landed"] and self.recv[vs]["fenced"],
                           "PV(%s) issued before chunks 0-3 landed (and, loaded by cp.async, were fenced)", j)
                self.check(self.own[os_]["tile"] == j and self.own[os_]["landed"] and self.own[os_]["fenced"],
                           "PV(%s) issued before chunks 4-7 landed and were fenced", j)

                def done():
                    self.recv[vs]["pv_read"] = True
                    self.own[os_]["pv_read"] = True
                    self.pslot[slot]["pv_read"] = True
                    self.pv_done_tiles.add(j)
                    self.b(0, "v_free", vs).arrive()
                    self.b(1, "v_free", vs).arrive()
                    self.b(1, "own_free", os_).arrive()
                    self.b(0, "p_free", slot).arrive()
                    self.b(1, "p_free", slot).arrive()
                    self.b(1, "pv_done", slot).arrive()
                    if j == self.n - 1:
                        self.b(1, "o_final", 0).arrive()
                self.later(done, fifo=("PV",))
            yield ("do", issue)

    def epilogue(self):
        yield self.W(1, "o_final", 0, 0)
        yield self.W(1, "fin_l", 0, 0)
        yield ("do", lambda: self.check(len(self.pv_done_tiles) == self.n, "epilogue before the last PV"))

    # ------------------------------------------------------------ scheduler
    def passed(self, cta, name, i, t, who):
        """A non-blocking parity probe (test_wait) for phase t."""
        bar = self.b(cta, name, i)
        if (bar.done & 1) != (t & 1):
            if bar.done != t + 1:
                raise ProtocolError("aliased probe of %s by %s: %d phases done, target phase %d"
                                    % (bar.name, who, bar.done, t))
            return True
        if bar.done > t + 1:
            raise ProtocolError("%s probes %s for phase %d, already %d done" % (who, bar.name, t, bar.done))
        return False

    def run(self):
        roles = {"q": self.q_load(), "fwd0": self.score_forwarder(),
                 "recv": self.recv_warp(), "vmax": self.value_max(), "pv": self.pv_issuer(),
                 "epi": self.epilogue()}
        if not self.decoupled:
            roles["fwd1"] = self.value_forwarder()
        for g in (0, 1):
            roles["sp%d" % g] = self.score_producers(g)
            roles["vp%d" % g] = self.value_producers(g)
            roles["sm%d" % g] = self.softmax(g)
        if self.decoupled:
            roles["vp2"] = self.value_recv_producers()
        for b in range(K_SBUF):
            for p in range(K_SPARTS):
                roles["s%d%d" % (b, p)] = self.s_issuer(b, p)
        cur = {name: None for name in roles}
        finished = set()
        steps = 0
        idle_polls = 0
        while True:
            steps += 1
            if steps > 2_000_000:
                raise ProtocolError("no progress")
            runnable = []
            for name, gen in roles.items():
                if name in finished:
                    continue
                if cur[name] is None:
                    try:
                        cur[name] = next(gen)
                    except StopIteration:
                        finished.add(name)
                        continue
                op = cur[name]
                if op[0] == "cond":
                    if op[1]():
                        runnable.append(name)
                elif op[0] == "wait":
                    _, cta, bname, i, t = op
                    bar = self.b(cta, bname, i)
                    if (bar.done & 1) != (t & 1):
                        if bar.done != t + 1:
                            raise ProtocolError("aliased wait on %s by %s: %d phases done, target phase %d"
                                                % (bar.name, name, bar.done, t))
                        runnable.append(name)
                    elif bar.done > t + 1:
                        raise ProtocolError("%s waits on %s for phase %d, already %d done"
                                            % (name, bar.name, t, bar.done))
                else:
                    runnable.append(name)
            busy = [n for n in runnable if cur[n][0] != "yield"]
            polling = [n for n in runnable if cur[n][0] == "yield"]
            if not busy and not self.delayed:
                if len(finished) == len(roles):
                    return
                idle_polls += 1
                if not polling or idle_polls > 8 * len(polling):
                    stuck = ", ".join("%s:%s" % (n, cur[n][:5] if cur[n] else None)
                                      for n in roles if n not in finished)
                    raise ProtocolError("deadlock: " + stuck)
                name = self.rng.choice(polling)
                cur[name] = None       # re-poll
                continue
            idle_polls = 0
            self.clock += 1
            ready = [i for i, (t, _) in enumerate(self.delayed) if t <= self.clock]
            if self.delayed and not busy and not ready:
                self.clock = min(t for t, _ in self.delayed)
                continue
            if ready and (not busy or self.rng.random() < 0.5):
                _, item = self.delayed.pop(self.rng.choice(ready))
                self._deliver(item)
                continue
            # a polling role re-polls only now and then
            pool = busy + [n for n in polling if self.rng.random() < 0.2]
            name = self.rng.choice(pool)
            op = cur[name]
            cur[name] = None
            if op[0] == "do":
                op[1]()
            # a passed wait needs nothing more; a "yield" lets the polling role retry


# planted mistakes, and the protocol form each applies to (None: both)
MUTATIONS = {"producers_uncoupled": None, "kv_full_without_fence": None, "producers_skip_stage_free": None,
             "issuers_skip_s_free": None, "softmax_skips_m_pub": None, "softmax_skips_p_free": None,
             "recv_skips_own_rows": None, "recv_producers_skip_slot_free": True, "recv_skips_v_full": True}


def run(ntiles, seed, mutation=None, decoupled=True):
    Model(ntiles, seed, mutation=mutation, decoupled=decoupled).run()
