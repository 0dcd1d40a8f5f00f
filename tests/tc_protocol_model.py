"""Discrete-event model of the tensor-memory GEMM kernel's barrier protocol.

The kernel's roles (weight producer, activation producer, one MMA issuer per strip of a
two-strip work unit, four dequant warpgroups and their shared epilogue) hand work to each
other through mbarriers in shared memory.  A parity wait on an mbarrier only tells the phase it
names from the phase just before it, so a wait that runs while the barrier is two phases
behind passes at once.  Whether that can happen depends on the order in which the roles' waits
and the asynchronous work (copies landing, multiplies completing) interleave, which a GPU run
samples only at its own timing.

This model restates each role's loop of gemm_tc_kernel (its waits, arrivals, copies, multiplies
and commits, in the kernel's order) and runs it under random interleavings.  Each step is one
role's next action or the completion of one asynchronous operation, taken uniformly among those
that can proceed.  It checks after every step:
  * every parity wait that passes finds the phase it meant completed (no aliasing);
  * no barrier gets more arrivals than its count in one phase;
  * a multiply reads the activation stage and A buffer of its own chunk, and its accumulator
    only after the previous segment was read out;
  * nothing overwrites a stage or A buffer that a multiply or a reader still needs;
  * each segment's read-out sees all of that segment's multiplies completed;
  * the run ends (no role is left waiting).

Roles, as in the kernel: a unit holds US strips (2, or 1 in the wide mode for large M).  Warpgroup
w of the dequant warps serves strip s = w % US of each unit and the chunks gs with
gs % (4 / US) == w // US of that strip (gs = unit * CH + chunk); strip s's issuer (one warp, in
chunk order) waits for a chunk's A buffer, then for its activation stage.

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
    NA: int          # A buffers per strip in tensor memory
    NS: int          # activation stages
    CH: int          # 128-row chunks per unit
    SW: int          # weight stages
    nunits: int      # units of this CTA
    KU: int          # units per strip pair
    kt0: int = 0     # unit index within its strip pair of the CTA's first unit
    idle_wempty: bool = True   # dequant warpgroups without a chunk in a unit do not touch its stage
    dequant_consumed_wait: bool = True  # the dequant waits for the A buffer's previous multiplies
    dequant_afull_wait: bool = False    # the dequant (instead of the issuer) waits for the chunk's
                                        # activation stage before signalling the chunk
    US: int = 2      # strips per unit: 2, or 1 (wide mode: four warpgroups on one strip)

    @property
    def nch(self):
        return self.nunits * self.CH

    @property
    def wreaders(self):
        return min(4, self.CH * self.US)  # warpgroups that read each unit's weight stage

    @property
    def ranks(self):
        return 4 // self.US               # warpgroups per strip


class Model:
    def __init__(self, cfg: Config):
        c = self.cfg = cfg
        self.wfull = [Barrier(f"wfull[{s}]", 1) for s in range(c.SW)]
        self.wempty = [Barrier(f"wempty[{s}]", 4 * c.wreaders) for s in range(c.SW)]
        self.afull = [Barrier(f"afull[{a}]", 1) for a in range(c.NS)]
        self.aempty = [Barrier(f"aempty[{a}]", c.US) for a in range(c.NS)]
        self.cfull = [[Barrier(f"cfull[{s}][{a}]", 4) for a in range(c.NA)] for s in range(2)]
        self.consumed = [[Barrier(f"consumed[{s}][{a}]", 1) for a in range(c.NA)] for s in range(2)]
        self.dfull = Barrier("dfull", c.US)
        self.dempty = Barrier("dempty", 16)
        self.w_content = {}        # weight stage -> unit whose copy landed there
        self.w_reads = {}          # unit -> dequant warps that have read it
        self.a_content = {}        # activation stage -> chunk whose copy landed there
        self.a_inflight = {}       # activation stage -> chunk whose copy is in flight
        self.decoded = [{}, {}]    # per strip: A buffer -> chunk decoded into it
        self.mma_done = [set(), set()]  # per strip: chunks whose multiplies completed
        self.epi_reads = {}        # segment -> warpgroups that have read it out
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
                self.require(self.w_reads.get(it - c.SW, 0) == 4 * c.wreaders,
                             f"weight copy of unit {it} overwrites stage {s} before unit {it - c.SW} was read")
            yield ("copy", self.wfull[s], lambda s=s, it=it: self.w_content.__setitem__(s, it))

    def act_producer(self):
        c = self.cfg
        for gs in range(c.nch):
            a = gs % c.NS
            if gs >= c.NS:
                yield ("wait", self.aempty[a], gs // c.NS - 1)
                self.require(all(gs - c.NS in self.mma_done[t] for t in range(c.US)),
                             f"activation copy of chunk {gs} overwrites stage {a} while chunk {gs - c.NS} is "
                             f"multiplied")
            self.a_inflight[a] = gs

            def land(a=a, gs=gs):
                self.a_content[a] = gs
            yield ("copy", self.afull[a], land)

    def issuer(self, s):
        c = self.cfg
        segs, first, kt = 0, True, c.kt0
        for it in range(c.nunits):
            seg_end = kt == c.KU - 1 or it == c.nunits - 1
            for cc in range(c.CH):
                gs = it * c.CH + cc
                a, st = gs % c.NA, gs % c.NS
                yield ("wait", self.cfull[s][a], gs // c.NA)
                if not c.dequant_afull_wait:
                    yield ("wait", self.afull[st], gs // c.NS)
                if first and segs > 0:
                    yield ("wait", self.dempty, segs - 1)
                self.require(self.a_content.get(st) == gs and self.a_inflight.get(st) == gs,
                             f"multiply of chunk {gs} reads activation stage {st} holding chunk "
                             f"{self.a_content.get(st)} (copy in flight: {self.a_inflight.get(st)})")
                self.require(self.decoded[s].get(a) == gs,
                             f"strip {s}: multiply of chunk {gs} reads A buffer {a} holding chunk "
                             f"{self.decoded[s].get(a)}")
                if first and segs > 0:
                    self.require(self.epi_reads.get(segs - 1, 0) == 4,
                                 f"strip {s}: chunk {gs} restarts the accumulator before segment {segs - 1} was "
                                 f"read out")
                yield ("mma", s, gs)
                yield ("commit", s, self.consumed[s][a])
                yield ("commit", s, self.aempty[st])
                first = False
            if seg_end:
                yield ("commit", s, self.dfull)
                segs, first = segs + 1, True
            kt = (kt + 1) % c.KU

    def warpgroup(self, w):
        c = self.cfg
        s, r = w % c.US, w // c.US
        segs, kt = 0, c.kt0
        for it in range(c.nunits):
            ws = it % c.SW
            seg_end = kt == c.KU - 1 or it == c.nunits - 1
            mine = [gs for gs in range(it * c.CH, (it + 1) * c.CH) if gs % c.ranks == r]
            if mine or not c.idle_wempty:
                yield ("wait", self.wfull[ws], it // c.SW)
                self.require(self.w_content.get(ws) == it, f"warpgroup {w} reads unit {it} from stage {ws} holding "
                                                           f"unit {self.w_content.get(ws)}")
                self.w_reads[it] = self.w_reads.get(it, 0) + 4
                yield ("arrive", self.wempty[ws], 4)
            for gs in mine:
                a = gs % c.NA
                if gs >= c.NA and c.dequant_consumed_wait:
                    yield ("wait", self.consumed[s][a], gs // c.NA - 1)
                if gs >= c.NA:
                    self.require(gs - c.NA in self.mma_done[s],
                                 f"strip {s}: decode of chunk {gs} overwrites A buffer {a} while chunk {gs - c.NA} "
                                 f"is multiplied")
                self.decoded[s][a] = gs
                if c.dequant_afull_wait:
                    yield ("wait", self.afull[gs % c.NS], gs // c.NS)
                yield ("arrive", self.cfull[s][a], 4)
            if seg_end:
                yield ("wait", self.dfull, segs)
                lo, hi = self.segments[segs]
                pending = [(t, g) for t in range(c.US) for g in range(lo, hi) if g not in self.mma_done[t]]
                self.require(not pending, f"read-out of segment {segs} while {pending} are still multiplied")
                self.epi_reads[segs] = self.epi_reads.get(segs, 0) + 1
                yield ("arrive", self.dempty, 4)
                segs += 1
            kt = (kt + 1) % c.KU

    # ---- scheduler ------------------------------------------------------------------------
    def run(self, rng: random.Random, max_steps: int = 400000):
        roles = [self.weight_producer(), self.act_producer()] + [self.issuer(s) for s in range(self.cfg.US)]
        roles += [self.warpgroup(w) for w in range(4)]
        nxt = {}
        for r in roles:
            self._advance(r, nxt)
        copies = []                                   # (barrier, on-land) in flight
        fifos = {s: deque() for s in range(self.cfg.US)}  # per issuer: multiplies and commits, in order
        for _ in range(max_steps):
            choices = []
            for r, act in nxt.items():
                if act[0] != "wait" or act[1].parity_passes(act[2]):
                    choices.append(("role", r))
            choices += [("copy", j) for j in range(len(copies))]
            choices += [("fifo", s) for s, q in fifos.items() if q]
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
                    self.mma_done[x].add(item[1])
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
