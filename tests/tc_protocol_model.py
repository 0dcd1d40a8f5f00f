"""Discrete-event model of the tensor-memory GEMM kernel's barrier protocol.

The kernel's roles (weight producer, two activation producers, NI MMA issuers, two dequant
teams and the epilogue) hand work to each other through mbarriers in shared memory.  A parity
wait on an mbarrier only tells the phase it names from the phase just before it, so a wait that
runs while the barrier is two phases behind passes at once.  Whether that can happen depends on
the order in which the roles' waits and the asynchronous work (copies landing, multiplies
completing) interleave, which a GPU run samples only at its own timing.

This model restates each role's loop of gemm_tc_kernel (its waits, arrivals, copies, multiplies
and commits, in the kernel's order) and runs it under random interleavings. Each step is one
role's next action or the completion of one asynchronous operation, taken uniformly among those
that can proceed.  It checks after every step:
  * every parity wait that passes finds the phase it meant completed (no aliasing);
  * no barrier gets more arrivals than its count in one phase;
  * a multiply reads the activation stage and A buffer of its own chunk, and its accumulator
    only after the previous segment was read out;
  * nothing overwrites a stage or A buffer that a multiply or a reader still needs;
  * each segment's read-out sees all of that segment's multiplies completed;
  * the run ends (no role is left waiting).

The model is host-side test code; switches select variants of the protocol, so the tests can
show that the checks catch the orderings that are wrong.
"""
from __future__ import annotations

import random
from collections import deque
from dataclasses import dataclass


class ProtocolError(AssertionError):
    pass


class Barrier:
    """mbarrier: an arrival count per phase plus a transaction count; phase = phases completed."""

    def __init__(self, name: str, count: int):
        self.name, self.count = name, count
        self.pending, self.tx, self.phase = count, 0, 0

    def arrive(self, n: int = 1):
        self.pending -= n
        if self.pending < 0:
            raise ProtocolError(f"{self.name}: {n} arrival(s) beyond the count in phase {self.phase}")
        self._advance()

    def expect_tx(self, n: int):
        self.tx += n

    def complete_tx(self, n: int):
        self.tx -= n
        if self.tx < 0:
            raise ProtocolError(f"{self.name}: transaction count below zero in phase {self.phase}")
        self._advance()

    def _advance(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def parity_passes(self, k: int) -> bool:
        # try_wait.parity with the parity of phase k: true once the phase in progress has the
        # other parity (phase k complete -- or, ambiguously, phase k - 1 still in progress)
        return (self.phase & 1) != (k & 1)


@dataclass
class Config:
    NA: int          # A buffers in tensor memory (activation stages too, unless `decoupled`)
    NI: int          # MMA issuers
    CH: int          # 128-row chunks per unit
    SW: int          # weight stages
    nunits: int      # units of this CTA
    KU: int          # units per strip
    kt0: int = 0     # unit index within its strip of the CTA's first unit
    NAS: int = 0     # activation stages when `decoupled` (0: = NA)
    decoupled: bool = False   # activation ring with its own empty barriers and a second commit
    afull_first: bool = False  # issuer waits for the activations before the A chunk
    idle_wait: bool = True     # an issuer without a chunk in a segment waits for the last read-out

    def __post_init__(self):
        if not self.NAS:
            self.NAS = self.NA

    @property
    def nch(self):
        return self.nunits * self.CH


class Model:
    def __init__(self, cfg: Config):
        c = self.cfg = cfg
        self.wfull = [Barrier(f"wfull[{s}]", 1) for s in range(c.SW)]
        self.wempty = [Barrier(f"wempty[{s}]", 16) for s in range(c.SW)]
        self.afull = [Barrier(f"afull[{a}]", 1) for a in range(c.NAS)]
        self.aempty = [Barrier(f"aempty[{a}]", 1) for a in range(c.NAS)]
        self.cfull = [Barrier(f"cfull[{a}]", 8) for a in range(c.NA)]
        self.consumed = [Barrier(f"consumed[{a}]", 1) for a in range(c.NA)]
        self.dfull = Barrier("dfull", c.NI)
        self.dempty = Barrier("dempty", 8)
        self.w_content = {}        # weight stage -> unit whose copy landed there
        self.w_reads = {}          # unit -> dequant warps that have read it
        self.a_content = {}        # activation stage -> chunk whose copy landed there
        self.a_inflight = {}       # activation stage -> chunk whose copy is in flight
        self.decoded = {}          # A buffer -> chunk decoded into it
        self.mma_done = set()      # chunks whose multiplies completed
        self.epi_done = 0          # segments read out
        # segments of this CTA: [first chunk, last chunk + 1)
        self.segments = []
        start, kt = 0, c.kt0
        for it in range(c.nunits):
            if kt == c.KU - 1 or it == c.nunits - 1:
                self.segments.append((start * c.CH, (it + 1) * c.CH))
                start = it + 1
            kt = (kt + 1) % c.KU

    def require(self, ok: bool, msg: str):
        if not ok:
            raise ProtocolError(msg)

    # ---- roles, in the kernel's order of waits and arrivals --------------------------------
    def weight_producer(self):
        c = self.cfg
        for it in range(c.nunits):
            s = it % c.SW
            if it >= c.SW:
                yield ("wait", self.wempty[s], it // c.SW - 1)
                self.require(self.w_reads.get(it - c.SW, 0) == 16,
                             f"weight copy of unit {it} overwrites stage {s} before unit {it - c.SW} was read")
            yield ("copy", self.wfull[s], lambda s=s, it=it: self.w_content.__setitem__(s, it))

    def act_producer(self, p):
        c = self.cfg
        for gc in range(p, c.nch, 2):
            a = gc % c.NAS
            if gc >= c.NAS:
                yield ("wait", (self.aempty if c.decoupled else self.consumed)[a], gc // c.NAS - 1)
                self.require(gc - c.NAS in self.mma_done,
                             f"activation copy of chunk {gc} overwrites stage {a} while chunk {gc - c.NAS} is multiplied")
            self.a_inflight[a] = gc

            def land(a=a, gc=gc):
                self.a_content[a] = gc
            yield ("copy", self.afull[a], land)

    def issuer(self, i):
        c = self.cfg
        segs, first, kt = 0, True, c.kt0
        for it in range(c.nunits):
            seg_end = kt == c.KU - 1 or it == c.nunits - 1
            for cc in range((i - it * c.CH) % c.NI, c.CH, c.NI):
                gc = it * c.CH + cc
                a, sa = gc % c.NA, gc % c.NAS
                waits = [("wait", self.cfull[a], gc // c.NA), ("wait", self.afull[sa], gc // c.NAS)]
                if c.afull_first:
                    waits.reverse()
                for w in waits:
                    yield w
                if first and segs > 0:
                    yield ("wait", self.dempty, segs - 1)
                self.require(self.a_content.get(sa) == gc and self.a_inflight.get(sa) == gc,
                             f"multiply of chunk {gc} reads activation stage {sa} holding chunk "
                             f"{self.a_content.get(sa)} (copy in flight: {self.a_inflight.get(sa)})")
                self.require(self.decoded.get(a) == gc,
                             f"multiply of chunk {gc} reads A buffer {a} holding chunk {self.decoded.get(a)}")
                if first:
                    self.require(self.epi_done >= segs,
                                 f"chunk {gc} restarts issuer {i}'s accumulator before segment {segs - 1} was read out")
                yield ("mma", i, gc)
                yield ("commit", i, self.consumed[a])
                if c.decoupled:
                    yield ("commit", i, self.aempty[sa])
                first = False
            if seg_end:
                if c.idle_wait and first and segs > 0:
                    yield ("wait", self.dempty, segs - 1)
                yield ("commit", i, self.dfull)
                segs, first = segs + 1, True
            kt = (kt + 1) % c.KU

    def team(self, t):
        c = self.cfg
        tcount, reuse_from = 0, (c.NA - t + 1) // 2
        segs, kt = 0, c.kt0
        for it in range(c.nunits):
            s = it % c.SW
            seg_end = kt == c.KU - 1 or it == c.nunits - 1
            yield ("wait", self.wfull[s], it // c.SW)
            self.require(self.w_content.get(s) == it, f"team {t} reads unit {it} from stage {s} holding unit "
                                                      f"{self.w_content.get(s)}")
            self.w_reads[it] = self.w_reads.get(it, 0) + 8
            yield ("arrive", self.wempty[s], 8)
            c0 = ((t ^ it) & 1) if c.CH & 1 else t
            for cc in range(c0, c.CH, 2):
                gc = it * c.CH + cc
                a = gc % c.NA
                if tcount >= reuse_from:
                    yield ("wait", self.consumed[a], gc // c.NA - 1)
                if gc >= c.NA:
                    self.require(gc - c.NA in self.mma_done,
                                 f"decode of chunk {gc} overwrites A buffer {a} while chunk {gc - c.NA} is multiplied")
                self.decoded[a] = gc
                yield ("arrive", self.cfull[a], 8)
                tcount += 1
            if seg_end and t == 0:
                yield ("wait", self.dfull, segs)
                lo, hi = self.segments[segs]
                pending = [g for g in range(lo, hi) if g not in self.mma_done]
                self.require(not pending, f"read-out of segment {segs} while chunks {pending} are still multiplied")
                self.epi_done += 1
                yield ("arrive", self.dempty, 8)
            if seg_end:
                segs += 1
            kt = (kt + 1) % c.KU

    # ---- scheduler ------------------------------------------------------------------------
    def run(self, rng: random.Random, max_steps: int = 200000):
        c = self.cfg
        roles = [self.weight_producer(), self.act_producer(0), self.act_producer(1)]
        roles += [self.issuer(i) for i in range(c.NI)] + [self.team(0), self.team(1)]
        nxt = {}
        for r in roles:
            self._advance(r, nxt)
        copies = []                                   # (barrier, on-land) in flight
        fifos = {i: deque() for i in range(c.NI)}     # per issuer: multiplies and commits, in order
        for _ in range(max_steps):
            choices = []
            for r, act in nxt.items():
                if act[0] != "wait" or act[1].parity_passes(act[2]):
                    choices.append(("role", r))
            choices += [("copy", j) for j in range(len(copies))]
            choices += [("fifo", i) for i, q in fifos.items() if q]
            if not choices:
                if nxt:
                    stuck = ", ".join(f"{a[1].name} phase {a[2]}" for a in nxt.values() if a[0] == "wait")
                    raise ProtocolError(f"deadlock: roles waiting on {stuck}")
                return
            kind, x = rng.choice(choices)
            if kind == "copy":
                bar, land = copies.pop(x)
                land()
                bar.complete_tx(1)
            elif kind == "fifo":
                item = fifos[x].popleft()
                if item[0] == "mma":
                    self.mma_done.add(item[1])
                else:
                    item[1].arrive(1)
            else:
                act = nxt[x]
                if act[0] == "wait":
                    bar, k = act[1], act[2]
                    self.require(bar.phase > k, f"parity wait on {bar.name} for phase {k} passed while phase "
                                                f"{bar.phase} was in progress")
                elif act[0] == "arrive":
                    act[1].arrive(act[2])
                elif act[0] == "copy":
                    act[1].expect_tx(1)
                    act[1].arrive(1)
                    copies.append((act[1], act[2]))
                elif act[0] == "mma":
                    fifos[act[1]].append(("mma", act[2]))
                elif act[0] == "commit":
                    fifos[act[1]].append(("commit", act[2]))
                self._advance(x, nxt)
        raise ProtocolError("step limit reached")

    @staticmethod
    def _advance(role, nxt):
        try:
            nxt[role] = next(role)
        except StopIteration:
            nxt.pop(role, None)


def explore(cfg: Config, seeds: int, seed0: int = 0):
    """Run `seeds` random interleavings; returns the first ProtocolError message, or None."""
    for sd in range(seed0, seed0 + seeds):
        try:
            Model(cfg).run(random.Random(sd))
        except ProtocolError as e:
            return f"seed {sd}: {e}"
    return None
