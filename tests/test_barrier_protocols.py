"""Models of the kernels' mbarrier hand-off protocols, run on the CPU under
random schedules.

Each kernel's roles (TMA producer, MMA issuer, gate and copy warps, and every
softmax / compute warp on its own, since each warp arrives on a barrier by
itself) are written as generators that yield the same waits, arrivals, loads,
MMAs and commits, in the same order, as the CUDA code.  TMA loads land in any
order; the tensor core runs one CTA's MMAs and commits in issue order (a
commit arrives once everything issued before it has run).  Every role, the
loads and the tensor core get a random speed per schedule, so that any of
them may run far ahead of the others.

Every shared-memory tile and TMEM region carries a tag naming what it holds
(K(3), S(1,2), P(1,2), dS(5), O(0,4), ...).  An access names the tag it
expects, so a schedule in which the tensor core reads a tile before its load
landed, overwrites S before the softmax read it, or accumulates into O before
the softmax rescaled it, fails.  The barriers check what the hardware cannot:

* every arrival belongs to the phase it was meant for (an early arrival would
  complete the wrong phase);
* a parity wait for phase p is evaluated only while the barrier is at phase
  p or p + 1 (two phases on, the parity answers wrongly);
* no schedule deadlocks, and the CTA never exits with a load or an MMA in
  flight (TMEM and shared memory are released at exit).

The planted-mistake cases at the end change one step of a model and must
fail, which shows the checks would catch such a change: the dQ gate's first
design (it ended in a launch failure on the GPU), the dQ kernel without its
PF handshake (the model found that gap), a forward S(j+1) issued before P(j)
was consumed, a rescale of O without waiting for P V, dK issued before dS^T
was written, and a ring load without its empty-slot wait.
"""
import random
from collections import deque

import pytest


class ProtocolError(AssertionError):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase = name, count, count, 0

    def arrive(self, n, phase):
        if phase != self.phase:
            raise ProtocolError(f"{self.name}: arrival for phase {phase} at phase {self.phase}")
        self.pending -= n
        if self.pending < 0:
            raise ProtocolError(f"{self.name}: too many arrivals in phase {phase}")
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, phase):
        # the hardware's parity wait answers correctly only at phase p (still
        # open) or p + 1 (completed): two phases on, or one phase short (the
        # completed phase p - 2 has p's parity), it answers wrongly
        if self.phase > phase + 1 or self.phase < phase:
            raise ProtocolError(f"{self.name}: wait for phase {phase} at phase {self.phase}")
        return self.phase > phase


class Cta:
    """Barriers, buffer tags, loads in flight and the tensor core's queues:
    one per issuing thread, each run in order (a commit arrives once
    everything its thread issued before it has run), the queues of two
    issuing threads interleaved in any order."""

    def __init__(self, bars):
        self.bars = {n: Bar(n, c) for n, c in bars.items()}
        self.mem = {}
        self.inflight = set()
        self.loads = []
        self.tcq = {}

    def tc_busy(self):
        return any(self.tcq.values())

    def read(self, reads, who):
        for buf, tag in reads.items():
            if buf in self.inflight:
                raise ProtocolError(f"{who}: reads {buf} while a load into it is in flight")
            if self.mem.get(buf) != tag:
                raise ProtocolError(f"{who}: {buf} holds {self.mem.get(buf)}, expected {tag}")

    def write(self, writes, who):
        for buf, tag in writes.items():
            if buf in self.inflight:
                raise ProtocolError(f"{who}: writes {buf} while a load into it is in flight")
            self.mem[buf] = tag

    def step(self, who, op):
        """Carry out a role's op; False when it is a wait that must repeat."""
        kind = op[0]
        if kind == "wait":
            try:
                return self.bars[op[1]].done(op[2])
            except ProtocolError as e:
                raise ProtocolError(f"{who}: {e}") from None
        if kind == "arrive":
            self.bars[op[1]].arrive(op[2], op[3])
        elif kind == "load":
            _, bar, phase, writes = op
            for buf in writes:
                if buf in self.inflight:
                    raise ProtocolError(f"{who}: second load into {buf}")
                self.inflight.add(buf)
            self.loads.append((bar, phase, writes))
        elif kind in ("mma", "commit"):
            self.tcq.setdefault(who, deque()).append(op)
        elif kind == "read":
            self.read(op[1], who)
        elif kind == "write":
            self.write(op[1], who)
        else:
            raise ValueError(op)
        return True

    def land(self, i):
        bar, phase, writes = self.loads.pop(i)
        for buf, tag in writes.items():
            self.inflight.discard(buf)
            self.mem[buf] = tag
        self.bars[bar].arrive(1, phase)

    def run_tc(self, rnd):
        op = self.tcq[rnd.choice(sorted(w for w, q in self.tcq.items() if q))].popleft()
        if op[0] == "commit":
            self.bars[op[1]].arrive(1, op[2])
        else:
            _, name, reads, writes = op
            self.read(reads, name)
            self.write(writes, name)


def simulate(model, seed, max_steps=500000):
    """model(rnd) -> (barrier counts, {role: generator}); rnd draws the
    data-dependent choices (whether a row's reference maximum moves)."""
    rnd = random.Random(seed)
    bars, roles = model(random.Random(seed + 1000003))
    cta = Cta(bars)
    # every role, the loads and the tensor core get their own speed, so that
    # any of them may run far ahead of the others
    speed = {r: rnd.choice((0.05, 0.3, 1.0)) for r in sorted(roles)}
    p_load, p_tc = rnd.choice((0.05, 0.3, 1.0)), rnd.choice((0.05, 0.3, 1.0))
    cur = {}
    for r, g in roles.items():
        op = next(g, None)
        if op is not None:
            cur[r] = op
    for _ in range(max_steps):
        if not cur:
            if cta.tc_busy() or cta.loads:
                raise ProtocolError(f"exit with work in flight: {cta.tcq} {cta.loads[:2]}")
            return
        progressed = False
        for r in rnd.sample(sorted(cur), len(cur)):
            if rnd.random() >= speed[r]:
                continue
            if cta.step(r, cur[r]):
                progressed = True
                op = next(roles[r], None)
                if op is None:
                    del cur[r]
                else:
                    cur[r] = op
        if cta.loads and rnd.random() < p_load:
            cta.land(rnd.randrange(len(cta.loads)))
            progressed = True
        if cta.tc_busy() and rnd.random() < p_tc:
            cta.run_tc(rnd)
            progressed = True
        if not progressed and not cta.tc_busy() and not cta.loads and all(
                op[0] == "wait" and not cta.step(r, op) for r, op in cur.items()):
            raise ProtocolError(f"deadlock: {cur}")
    raise ProtocolError("did not finish")


def each_seed(model, seeds=range(60)):
    for seed in seeds:
        simulate(model, seed)


def fails_on_some_seed(model, seeds=range(80)):
    for seed in seeds:
        try:
            simulate(model, seed)
        except ProtocolError:
            return True
    return False


def kv_ring_producer(n_blocks, nslot, first, tiles=("K", "V"), skip_empty=False):
    """The forward-style producer: Q, then K_j, V_j of every key block
    through one ring of nslot tiles; at exit it waits for its last loads."""
    last = {}
    yield ("load", "Q", 0, first)
    for j in range(n_blocks):
        for w, nm in enumerate(tiles):
            idx = 2 * j + w
            s = idx % nslot
            if not skip_empty:
                yield ("wait", f"E{s}", idx // nslot - 1)  # a slot's first use passes
            yield ("load", f"F{s}", idx // nslot, {f"kv{s}": f"{nm}({j})"})
            last[s] = idx // nslot
    yield ("wait", "Q", 0)
    for s, ph in last.items():
        yield ("wait", f"F{s}", ph)


def ring_bars(nslot):
    bars = {}
    for s in range(nslot):
        bars[f"F{s}"] = bars[f"E{s}"] = 1
    return bars


# ---------------------------------------------------------------- dQ kernel
def dq_model(nj, KS=3, VS=2, handshake=True, first_gate_design=False, two_issuers=False,
             single_dqd=False, skip_dqd=False, early_dp=False, dp_before_dq=False,
             late_ke=False):
    """Sixteen compute warps (w, q): key quarter w (32 columns of S, dP, its
    dS written into the first 16) and TMEM lanes 32q.. (query rows); each
    arrives on its own.  The MMA thread
    arrives on PFS once it has seen dS(j) complete; a warp waits for that
    before its dS(j+1) arrival, so PF is never a phase ahead of its waiter.
    two_issuers (a variant that was tried and measured slower, not the
    kernel's protocol): S and dP are issued by one thread, dQ by another (its
    own tensor-core queue); dQ(j) reads dS(j) in dP buffer j % 2, which dP(j+2)
    overwrites, so the dQ thread commits DQD(j % 2) after dQ(j) and the S/dP
    thread waits for it (phase j // 2) before dP(j+2); the dQ thread, which
    waits for PF, is the one that arrives on PFS.  single_dqd (one DQD
    barrier for both buffers) and skip_dqd are planted mistakes.

    early_dp: dP(j+2) is issued right after dQ(j), into the buffer dQ(j) has
    just read, instead of next to S(j+2) behind LD(j+1); only S(j+1) waits for
    LD(j), whose gate then folds in K_{j+1} alone, and the MMA thread waits
    for V_{j+2} itself.  The producer loads in the products' first-use order
    (K_0, V_0, V_1, K_1, V_2, K_2, ...).  late_ke: the commit that frees K_j's
    slot follows dP(j+2), so dQ(j) and dP(j+2) are issued back to back.
    dp_before_dq (dP(j+2) issued before dQ(j)) is a planted mistake."""
    warps = [(w, q) for w in range(4) for q in range(4)]

    def model(rnd):
        bars = {"QDO": 1, "SDF": 1, "LD": 513, "PF": 513 if first_gate_design else 512, "ACC": 1,
                "PFS": 1, "DQD0": 1, "DQD1": 1, "DONE": 1}
        for nm, ns in (("K", KS), ("V", VS)):
            for s in range(ns):
                bars[f"{nm}F{s}"] = bars[f"{nm}E{s}"] = 1

        def every(pre, tag):
            return {f"{pre}.{w}.{q}": tag for w, q in warps}

        def producer():
            yield ("load", "QDO", 0, dict(every("Q", "Q"), dO="dO"))
            last = {}
            for i in range(nj):
                order = (("V", VS), ("K", KS)) if early_dp and i > 0 else (("K", KS), ("V", VS))
                for nm, ns in order:
                    s = i % ns
                    yield ("wait", f"{nm}E{s}", i // ns - 1)
                    yield ("load", f"{nm}F{s}", i // ns, {f"{nm}{s}": f"{nm}({i})"})
                    last[f"{nm}F{s}"] = i // ns
            yield ("wait", "QDO", 0)
            for bar, ph in last.items():
                yield ("wait", bar, ph)

        def gate():
            for j in range(nj):
                if not early_dp and j > 0:
                    # V_{j+1}'s slot last held V_{j-1}: LD(j-1) says it landed, so
                    # the parity wait below cannot be a phase short (waiting V
                    # first, as an earlier form did, could be)
                    yield ("wait", "LD", j - 1)
                if j + 1 < nj:
                    yield ("wait", f"KF{(j + 1) % KS}", (j + 1) // KS)
                    if not early_dp:
                        yield ("wait", f"VF{(j + 1) % VS}", (j + 1) // VS)
                if early_dp and j > 0:
                    yield ("wait", "LD", j - 1)
                yield ("arrive", "LD", 1, j)
                if first_gate_design:
                    # it also held dS(j) back until V_{j+2} had landed
                    if j + 2 < nj:
                        yield ("wait", f"VF{(j + 2) % VS}", (j + 2) // VS)
                    if j > 0:
                        yield ("wait", "PF", j - 1)
                    yield ("arrive", "PF", 1, j)

        def copy():
            yield ("wait", "QDO", 0)
            yield ("read", {"dO": "dO"})

        def s_mma(jj):
            return ("mma", f"S({jj})", dict(every("Q", "Q"), **{f"K{jj % KS}": f"K({jj})"}),
                    every("S", f"S({jj})"))

        def dp_mma(jj):
            return ("mma", f"dP({jj})", {"dO": "dO", f"V{jj % VS}": f"V({jj})"},
                    every(f"DP{jj & 1}", f"dP({jj})"))

        def mma():
            yield ("wait", "QDO", 0)
            yield ("wait", "KF0", 0)
            yield s_mma(0)
            yield ("wait", "VF0", 0)
            yield dp_mma(0)
            yield ("commit", "VE0", 0)
            yield ("commit", "SDF", 0)
            if early_dp and nj > 1:
                yield ("wait", "VF1", 0)
                yield dp_mma(1)
                yield ("commit", f"VE{1 % VS}", 1 // VS)
            for j in range(nj):
                if early_dp:
                    if j + 1 < nj:
                        yield ("wait", "LD", j)
                        yield s_mma(j + 1)
                        yield ("commit", "SDF", j + 1)

                    def dp_next():
                        yield ("wait", f"VF{(j + 2) % VS}", (j + 2) // VS)
                        yield dp_mma(j + 2)  # over dS(j), which dQ(j) reads first
                        yield ("commit", f"VE{(j + 2) % VS}", (j + 2) // VS)
                    if dp_before_dq and j + 2 < nj:
                        yield from dp_next()
                    yield ("wait", "PF", j)
                    yield ("arrive", "PFS", 1, j)
                    yield dq_mma(j)
                    if not late_ke:
                        yield ("commit", f"KE{j % KS}", j // KS)
                    if not dp_before_dq and j + 2 < nj:
                        yield from dp_next()
                    if late_ke:
                        yield ("commit", f"KE{j % KS}", j // KS)
                    continue
                if j + 1 < nj:
                    yield ("wait", "LD", j)
                    yield s_mma(j + 1)
                    if two_issuers and j + 1 >= 2 and not skip_dqd:
                        # dQ(j-1), the last reader of dP buffer (j+1) % 2
                        if single_dqd:
                            yield ("wait", "DQD0", j - 1)
                        else:
                            yield ("wait", f"DQD{(j + 1) & 1}", (j - 1) >> 1)
                    yield dp_mma(j + 1)
                    yield ("commit", f"VE{(j + 1) % VS}", (j + 1) // VS)
                    yield ("commit", "SDF", j + 1)
                if two_issuers:
                    continue
                yield ("wait", "PF", j)
                if handshake:
                    yield ("arrive", "PFS", 1, j)
                yield dq_mma(j)
                yield ("commit", f"KE{j % KS}", j // KS)
            if two_issuers:
                yield ("commit", "DONE", 0)
                yield ("wait", "DONE", 0)
            else:
                yield ("commit", "ACC", 0)
                yield ("wait", "ACC", 0)

        def dq_mma(j):
            reads = dict(every(f"DP{j & 1}", f"dS({j})"), **{f"K{j % KS}": f"K({j})"})
            if j > 0:
                reads["dQ"] = f"dQ({j - 1})"
            return ("mma", f"dQ({j})", reads, {"dQ": f"dQ({j})"})

        def mma_dq():
            for j in range(nj):
                yield ("wait", "PF", j)
                if handshake:
                    yield ("arrive", "PFS", 1, j)
                yield dq_mma(j)
                yield ("commit", f"KE{j % KS}", j // KS)
                if single_dqd:
                    yield ("commit", "DQD0", j)
                else:
                    yield ("commit", f"DQD{j & 1}", j >> 1)
            yield ("commit", "ACC", 0)
            yield ("wait", "ACC", 0)

        def compute(w, q):
            me = f"{w}.{q}"
            for j in range(nj):
                yield ("wait", "SDF", j)
                yield ("read", {f"S.{me}": f"S({j})", f"DP{j & 1}.{me}": f"dP({j})"})
                yield ("arrive", "LD", 32, j)
                yield ("write", {f"DP{j & 1}.{me}": f"dS({j})"})
                if handshake and j > 0:
                    yield ("wait", "PFS", j - 1)
                yield ("arrive", "PF", 32, j)
            yield ("wait", "ACC", 0)
            yield ("read", {"dQ": f"dQ({nj - 1})"})
            yield ("write", {f"Q.{me}": "dQ out"})  # staging in the Q tile

        roles = {"prod": producer(), "gate": gate(), "copy": copy(), "mma": mma()}
        if two_issuers:
            roles["mmaq"] = mma_dq()
        for w, q in warps:
            roles[f"c{w}{q}"] = compute(w, q)
        return bars, roles

    return model


# -------------------------------------------------------------- dK/dV kernel
def dkdv_model(n_it, NST=2, dk_before_dsf=False, ds_smem=False, ds_in_do=True, skip_dvd=False,
               p_before_str=False, three_regions=False, early_dpt=False, skip_dsf_wait=False,
               late_ste=False):
    """Sixteen compute warps (g, q): query columns 32g.. of the transposed
    tiles (warpgroup g) and key rows 32q.. (TMEM lanes).  The kernel's
    protocol (ds_smem False): a warp forms P^T(it) as soon as S^T(it) is in
    TMEM (barrier STR) and writes it over the S^T columns it read (half 'p'),
    then, once dP^T(it) is in TMEM (SDF), copies dP^T(it) to registers (LD)
    and writes dS^T(it) over the other half ('d').  The MMA thread: dV(it)
    after P^T, S^T(it+1) over dP^T(it) after LD, dK(it) after dS^T, then
    dP^T(it+1) over P^T(it), dS^T(it).  three_regions (a variant tried at
    d = 64, where TMEM has a third 128-column region, and measured slower:
    dK/dV 0.551 -> 0.583 ms on gpt2s): the regions rotate, S^T(it) in
    R[it % 3] and dP^T(it) in R[(it + 1) % 3], so dP^T(it+1) goes into the
    region P^T, dS^T(it-1) left and is issued right after S^T(it+1), before
    dK(it).
    A warp then arrives on DSF(it) only once DSF(it-1) has completed (a fast
    warp could otherwise run a step ahead into the previous phase).
    early_dpt (that early issue with only two regions, over P^T(it), dS^T(it)),
    skip_dsf_wait (three regions without the DSF(it-1) wait) and p_before_str
    (P^T formed without waiting for S^T) are planted mistakes.  late_ste (a
    variant tried and measured slower: gqa8k dK/dV 2.84 -> 3.06 ms, the
    two-stage ring starved): the commit that frees the step's {Q, dO} stage
    follows dP^T(it+1) and its SDF commit, so dK(it) and dP^T(it+1) go to the
    tensor core back to back.  A variant that was tried and
    measured slower (ds_smem True, with the earlier single-step compute):
    dS^T goes to shared memory instead -- over the stage's dO tile (ds_in_do,
    d = 128) or into a buffer of its own (d = 64) -- once the MMA thread's
    DVD commit after dV(it) has completed, so dP^T(it+1) follows dV(it) and
    dK(it) reads dS^T from shared memory after it."""
    warps = [(g, q) for g in range(4) for q in range(4)]

    def model(rnd):
        bars = {"KV": 1, "SDF": 1, "LD": 512, "PF": 512, "DSF": 512, "ACC": 1, "DVD": 1,
                "STR": 1}
        for s in range(NST):
            bars[f"STF{s}"] = 1 + 32  # the load, and the 32 lanes' vector writes
            bars[f"STE{s}"] = 1

        def reg_s(it):  # S^T(it), then P^T(it) (/ dS^T(it))
            if three_regions:
                return "R%d" % (it % 3)
            return "Y" if it & 1 else "X"

        def reg_d(it):  # dP^T(it)
            if three_regions:
                return "R%d" % ((it + 1) % 3)
            return "X" if it & 1 else "Y"

        def region(r, tag):
            return {f"{r}.{g}.{q}.{c}": tag for g, q in warps for c in "pd"}

        def ds_buf(it, g, q):  # where warp (g, q) writes dS^T(it)
            if not ds_smem:
                return f"{reg_s(it)}.{g}.{q}.d"
            return f"dO{it % NST}.{g}.{q}" if ds_in_do else f"DS.{g}.{q}"

        def stage_load(it):
            tags = {f"Q{it % NST}": f"Q({it})"}
            tags.update({f"dO{it % NST}.{g}.{q}": f"dO({it})" for g, q in warps})
            return tags

        def producer():
            yield ("load", "KV", 0, {"K": "K", "V": "V"})
            last = {}
            for it in range(n_it):
                s = it % NST
                yield ("wait", f"STE{s}", it // NST - 1)
                yield ("load", f"STF{s}", it // NST, stage_load(it))
                yield ("write", {f"vec{s}": f"lse,D({it})"})
                yield ("arrive", f"STF{s}", 32, it // NST)
                last[s] = it // NST
            yield ("wait", "KV", 0)
            for s, ph in last.items():
                yield ("wait", f"STF{s}", ph)

        def st_mma(it):
            return ("mma", f"S^T({it})", {"K": "K", f"Q{it % NST}": f"Q({it})"},
                    region(reg_s(it), f"S^T({it})"))

        def dpt_mma(it):
            reads = {"V": "V"}
            reads.update({f"dO{it % NST}.{g}.{q}": f"dO({it})" for g, q in warps})
            return ("mma", f"dP^T({it})", reads, region(reg_d(it), f"dP^T({it})"))

        def dv_mma(it):
            reads = {f"{reg_s(it)}.{g}.{q}.p": f"P^T({it})" for g, q in warps}
            reads.update({f"dO{it % NST}.{g}.{q}": f"dO({it})" for g, q in warps})
            if it > 0:
                reads["dV"] = f"dV({it - 1})"
            return ("mma", f"dV({it})", reads, {"dV": f"dV({it})"})

        def dk_mma(it):
            reads = {ds_buf(it, g, q): f"dS^T({it})" for g, q in warps}
            reads[f"Q{it % NST}"] = f"Q({it})"
            if it > 0:
                reads["dK"] = f"dK({it - 1})"
            return ("mma", f"dK({it})", reads, {"dK": f"dK({it})"})

        def mma_two_step():
            yield ("wait", "KV", 0)
            yield ("wait", "STF0", 0)
            yield st_mma(0)
            yield ("commit", "STR", 0)
            yield dpt_mma(0)
            yield ("commit", "SDF", 0)
            for it in range(n_it):
                s, s2 = it % NST, (it + 1) % NST
                more = it + 1 < n_it
                yield ("wait", "PF", it)
                yield dv_mma(it)
                early = three_regions or early_dpt
                if more:
                    yield ("wait", f"STF{s2}", (it + 1) // NST)
                    yield ("wait", "LD", it)
                    yield st_mma(it + 1)  # over dP^T(it)
                    yield ("commit", "STR", it + 1)
                    if early:  # into the third region (P^T, dS^T(it-1) were read by dK(it-1))
                        yield dpt_mma(it + 1)
                        yield ("commit", "SDF", it + 1)
                if not dk_before_dsf:
                    yield ("wait", "DSF", it)
                yield dk_mma(it)
                if not late_ste:
                    yield ("commit", f"STE{s}", it // NST)
                if more and not early:
                    yield dpt_mma(it + 1)  # over P^T(it), dS^T(it)
                    yield ("commit", "SDF", it + 1)
                if late_ste:
                    yield ("commit", f"STE{s}", it // NST)
            yield ("commit", "ACC", 0)
            yield ("wait", "ACC", 0)

        def compute_two_step(g, q):
            me = f"{g}.{q}"
            for it in range(n_it):
                s = it % NST
                rs, rd = reg_s(it), reg_d(it)
                if not p_before_str:
                    yield ("wait", "STR", it)
                yield ("read", {f"{rs}.{me}.p": f"S^T({it})", f"{rs}.{me}.d": f"S^T({it})",
                                f"vec{s}": f"lse,D({it})"})
                yield ("write", {f"{rs}.{me}.p": f"P^T({it})"})
                yield ("arrive", "PF", 32, it)
                yield ("wait", "SDF", it)
                yield ("read", {f"{rd}.{me}.p": f"dP^T({it})", f"{rd}.{me}.d": f"dP^T({it})",
                                f"vec{s}": f"lse,D({it})"})
                yield ("arrive", "LD", 32, it)
                yield ("write", {ds_buf(it, g, q): f"dS^T({it})"})
                # with dP^T(it) issued before dK(it-1), a fast warp can reach
                # here while DSF(it-1) still waits for slow ones: it arrives only
                # once that phase has completed
                if three_regions and it > 0 and not skip_dsf_wait:
                    yield ("wait", "DSF", it - 1)
                yield ("arrive", "DSF", 32, it)
            yield ("wait", "ACC", 0)
            yield ("read", {"dV": f"dV({n_it - 1})", "dK": f"dK({n_it - 1})"})
            yield ("write", {"Q0": "out"})  # staging in stage 0's tiles

        def mma():
            yield ("wait", "KV", 0)
            yield ("wait", "STF0", 0)
            yield st_mma(0)
            yield dpt_mma(0)
            yield ("commit", "SDF", 0)
            for it in range(n_it):
                s, s2 = it % NST, (it + 1) % NST
                more = it + 1 < n_it
                if more:
                    yield ("wait", f"STF{s2}", (it + 1) // NST)
                    yield ("wait", "LD", it)
                    yield st_mma(it + 1)  # over dP^T(it)
                yield ("wait", "PF", it)
                yield dv_mma(it)
                if ds_smem:
                    yield ("commit", "DVD", it)
                    if more:
                        yield dpt_mma(it + 1)  # over P^T(it)
                        yield ("commit", "SDF", it + 1)
                if not dk_before_dsf:
                    yield ("wait", "DSF", it)
                yield dk_mma(it)
                yield ("commit", f"STE{s}", it // NST)
                if more and not ds_smem:
                    yield dpt_mma(it + 1)  # over P^T(it), dS^T(it)
                    yield ("commit", "SDF", it + 1)
            yield ("commit", "ACC", 0)
            yield ("wait", "ACC", 0)

        def compute(g, q):
            me = f"{g}.{q}"
            for it in range(n_it):
                s = it % NST
                rs, rd = reg_s(it), reg_d(it)
                yield ("wait", "SDF", it)
                yield ("read", {f"{rd}.{me}.p": f"dP^T({it})", f"{rd}.{me}.d": f"dP^T({it})",
                                f"vec{s}": f"lse,D({it})"})
                yield ("arrive", "LD", 32, it)
                yield ("read", {f"{rs}.{me}.p": f"S^T({it})", f"{rs}.{me}.d": f"S^T({it})"})
                yield ("write", {f"{rs}.{me}.p": f"P^T({it})"})
                yield ("arrive", "PF", 32, it)
                if ds_smem and not skip_dvd:
                    yield ("wait", "DVD", it)
                yield ("write", {ds_buf(it, g, q): f"dS^T({it})"})
                yield ("arrive", "DSF", 32, it)
            yield ("wait", "ACC", 0)
            yield ("read", {"dV": f"dV({n_it - 1})", "dK": f"dK({n_it - 1})"})
            yield ("write", {"Q0": "out"})  # staging in stage 0's tiles

        if ds_smem:
            roles = {"prod": producer(), "mma": mma()}
            for g, q in warps:
                roles[f"c{g}{q}"] = compute(g, q)
        else:
            roles = {"prod": producer(), "mma": mma_two_step()}
            for g, q in warps:
                roles[f"c{g}{q}"] = compute_two_step(g, q)
        return bars, roles

    return model


def dkdv_persistent_model(items, NST=3, mistake=None, lagging_store=False, kv_buffers=1):
    """The persistent dK/dV kernel (d = 64): one CTA walks `items`, each the
    query-step count of one (batch, kv head, 128-key block).  Steps carry
    global indices g across items, so the {Q, dO} stage ring, the TMEM
    regions (X/Y by g's parity) and the per-step barriers run on.  Within an
    item the order is the one-item kernel's two-step order.  K and V are
    reloaded once the item's last S^T and dP^T have read them (KVE: a commit
    after the item's last dP^T).  An item's first S^T goes over dP^T of the
    previous item's last step, so it waits for LD of that step.  dV and dK of
    the next item start afresh only after PF / DSF of its first step, which
    the warps arrive on after their epilogue's TMEM loads.  The warps stage
    dV and dK in a buffer of their own once the store warp has read the
    previous item's (EPE), and the store warp stores them (EPF).  (The
    cross-item LD wait is implied here: the MMA thread waited for DSF of that
    step, which every warp arrives on after LD; the kernel keeps it anyway.)
    lagging_store makes the store warp read an item's staging only after the
    next item's accumulators are done, the lag EPE exists for.  kv_buffers=2:
    item it's K, V go to buffer it % 2 (barriers KV, KVE per buffer), loaded
    once item it - 2 is done with that buffer, so the next item's tiles land
    while the current item runs.  mistake: "no_kve", "no_epe" drop the
    matching wait."""
    KB = kv_buffers
    warps = [(g, q) for g in range(4) for q in range(4)]
    starts = [sum(items[:i]) for i in range(len(items))]

    def model(rnd):
        bars = {"SDF": 1, "LD": 512, "PF": 512, "DSF": 512, "ACC": 1,
                "STR": 1, "EPF": 512, "EPE": 1, "DONE": 1}
        for b_ in range(KB):
            bars[f"KV{b_}"] = 1
            bars[f"KVE{b_}"] = 1
        for s_ in range(NST):
            bars[f"STF{s_}"] = 1 + 32
            bars[f"STE{s_}"] = 1

        def reg_s(g):
            return "Y" if g & 1 else "X"

        def reg_d(g):
            return "X" if g & 1 else "Y"

        def region(r, tag):
            return {f"{r}.{w}.{q}.{c}": tag for w, q in warps for c in "pd"}

        def producer():
            last = {}
            for it, n in enumerate(items):
                b = it % KB
                if it >= KB and mistake != "no_kve":
                    yield ("wait", f"KVE{b}", (it - KB) // KB)
                yield ("load", f"KV{b}", it // KB, {f"K{b}": f"K({it})", f"V{b}": f"V({it})"})
                for j in range(n):
                    g = starts[it] + j
                    sl = g % NST
                    yield ("wait", f"STE{sl}", g // NST - 1)
                    tags = {f"Q{sl}": f"Q({g})"}
                    tags.update({f"dO{sl}.{w}.{q}": f"dO({g})" for w, q in warps})
                    yield ("load", f"STF{sl}", g // NST, tags)
                    yield ("write", {f"vec{sl}": f"lse,D({g})"})
                    yield ("arrive", f"STF{sl}", 32, g // NST)
                    last[sl] = g // NST
            for b in range(KB):
                used = [i for i in range(len(items)) if i % KB == b]
                if used:
                    yield ("wait", f"KV{b}", used[-1] // KB)
            for sl, ph in last.items():
                yield ("wait", f"STF{sl}", ph)

        def st_mma(it, g):
            return ("mma", f"S^T({g})", {f"K{it % KB}": f"K({it})", f"Q{g % NST}": f"Q({g})"},
                    region(reg_s(g), f"S^T({g})"))

        def dpt_mma(it, g):
            reads = {f"V{it % KB}": f"V({it})"}
            reads.update({f"dO{g % NST}.{w}.{q}": f"dO({g})" for w, q in warps})
            return ("mma", f"dP^T({g})", reads, region(reg_d(g), f"dP^T({g})"))

        def dv_mma(it, j, g):
            reads = {f"{reg_s(g)}.{w}.{q}.p": f"P^T({g})" for w, q in warps}
            reads.update({f"dO{g % NST}.{w}.{q}": f"dO({g})" for w, q in warps})
            if j > 0:
                reads["dV"] = f"dV({it},{j - 1})"
            return ("mma", f"dV({g})", reads, {"dV": f"dV({it},{j})"})

        def dk_mma(it, j, g):
            reads = {f"{reg_s(g)}.{w}.{q}.d": f"dS^T({g})" for w, q in warps}
            reads[f"Q{g % NST}"] = f"Q({g})"
            if j > 0:
                reads["dK"] = f"dK({it},{j - 1})"
            return ("mma", f"dK({g})", reads, {"dK": f"dK({it},{j})"})

        def mma():
            for it, n in enumerate(items):
                g0 = starts[it]
                yield ("wait", f"KV{it % KB}", it // KB)
                yield ("wait", f"STF{g0 % NST}", g0 // NST)
                if it > 0 and mistake != "no_ld_cross":
                    yield ("wait", "LD", g0 - 1)  # S^T(g0) goes over dP^T(g0 - 1)
                yield st_mma(it, g0)
                yield ("commit", "STR", g0)
                yield dpt_mma(it, g0)
                yield ("commit", "SDF", g0)
                if n == 1:
                    yield ("commit", f"KVE{it % KB}", it // KB)
                for j in range(n):
                    g = g0 + j
                    more = j + 1 < n
                    yield ("wait", "PF", g)
                    yield dv_mma(it, j, g)
                    if more:
                        yield ("wait", f"STF{(g + 1) % NST}", (g + 1) // NST)
                        yield ("wait", "LD", g)
                        yield st_mma(it, g + 1)
                        yield ("commit", "STR", g + 1)
                    yield ("wait", "DSF", g)
                    yield dk_mma(it, j, g)
                    yield ("commit", f"STE{g % NST}", g // NST)
                    if more:
                        yield dpt_mma(it, g + 1)
                        yield ("commit", "SDF", g + 1)
                        if j + 2 == n:
                            yield ("commit", f"KVE{it % KB}", it // KB)  # the item's last S^T, dP^T
                yield ("commit", "ACC", it)
            yield ("commit", "DONE", 0)
            yield ("wait", "DONE", 0)

        def compute(w, q):
            me = f"{w}.{q}"
            for it, n in enumerate(items):
                for j in range(n):
                    g = starts[it] + j
                    sl = g % NST
                    rs, rd = reg_s(g), reg_d(g)
                    yield ("wait", "STR", g)
                    yield ("read", {f"{rs}.{me}.p": f"S^T({g})", f"{rs}.{me}.d": f"S^T({g})",
                                    f"vec{sl}": f"lse,D({g})"})
                    yield ("write", {f"{rs}.{me}.p": f"P^T({g})"})
                    yield ("arrive", "PF", 32, g)
                    yield ("wait", "SDF", g)
                    yield ("read", {f"{rd}.{me}.p": f"dP^T({g})", f"{rd}.{me}.d": f"dP^T({g})",
                                    f"vec{sl}": f"lse,D({g})"})
                    yield ("arrive", "LD", 32, g)
                    yield ("write", {f"{rs}.{me}.d": f"dS^T({g})"})
                    yield ("arrive", "DSF", 32, g)
                yield ("wait", "ACC", it)
                yield ("read", {"dV": f"dV({it},{n - 1})", "dK": f"dK({it},{n - 1})"})
                if it > 0 and mistake != "no_epe":
                    yield ("wait", "EPE", it - 1)
                yield ("write", {f"ST.{me}": f"out({it})"})
                yield ("arrive", "EPF", 32, it)

        def store():
            for it in range(len(items)):
                yield ("wait", "EPF", it)
                if lagging_store and it + 1 < len(items):
                    yield ("wait", "ACC", it + 1)
                yield ("read", {f"ST.{w}.{q}": f"out({it})" for w, q in warps})
                yield ("arrive", "EPE", 1, it)

        roles = {"prod": producer(), "mma": mma(), "store": store()}
        for w, q in warps:
            roles[f"c{w}{q}"] = compute(w, q)
        return bars, roles

    return model


def dq_persistent_model(items, KS=4, VS=3, copy_q=True, mistake=None, qdo_buffers=1):
    """The persistent dQ kernel (d = 64): one CTA walks `items`, each the key
    block count of one (batch, head, 128-query block).  Blocks carry global
    indices g across items, so the K/V rings, the dP buffers (g % 2) and the
    per-block barriers (SDF, LD, PF, PFS) run on from one item to the next.
    Within an item the order is the one-item kernel's (dP two blocks ahead).
    At an item's start the MMA thread waits for its Q, dO (QDO) and for LD of
    the previous item's last block before the new S(g0): the data is implied
    by PF, which it waited for, but without that wait its parity wait for
    LD(g0) could find the barrier a phase short.  The item's first dQ, which
    starts the accumulator afresh, follows PF(g0), and every warp arrives on
    that only after it has read the previous item's dQ out of TMEM.  Q and
    dO are free for the next item once its last S and dP are done and the
    copy warp has read dO (QE: a commit after the item's last S, one arrival
    from the copy warp).  The warps stage dQ in a buffer of its own, once the
    previous item's store has read it (EPE), and the copy warp, after the
    item's dO copy, stores it from there (EPF).  qdo_buffers=2: item it's Q,
    dO go to buffer it % 2 (barriers QDO, QE per buffer), loaded once item
    it - 2 is done with that buffer, so the next item's tiles land while the
    current item runs.  mistake: "no_qe", "no_ld_cross", "no_epe" drop the
    matching wait."""
    QB = qdo_buffers
    warps = [(w, q) for w in range(4) for q in range(4)]
    G = sum(items)
    starts = [sum(items[:i]) for i in range(len(items))]

    def model(rnd):
        bars = {"SDF": 1, "LD": 513, "PF": 512, "PFS": 1, "ACC": 1, "EPF": 512, "EPE": 1,
                "DONE": 1}
        for b_ in range(QB):
            bars[f"QDO{b_}"] = 1
            bars[f"QE{b_}"] = 1 + (1 if copy_q else 0)
        for nm, ns in (("K", KS), ("V", VS)):
            for s_ in range(ns):
                bars[f"{nm}F{s_}"] = bars[f"{nm}E{s_}"] = 1

        def every(pre, tag):
            return {f"{pre}.{w}.{q}": tag for w, q in warps}

        def producer():
            last = {}
            for it, nj in enumerate(items):
                b = it % QB
                if it >= QB and mistake != "no_qe":
                    yield ("wait", f"QE{b}", (it - QB) // QB)
                yield ("load", f"QDO{b}", it // QB,
                       dict(every(f"Q{b}", f"Q({it})"), **{f"dO{b}": f"dO({it})"}))
                g0 = starts[it]
                order = [("K", g0), ("V", g0)]
                for i in range(1, nj):
                    order += [("V", g0 + i), ("K", g0 + i)]
                for nm, g in order:
                    ns = KS if nm == "K" else VS
                    sl = g % ns
                    yield ("wait", f"{nm}E{sl}", g // ns - 1)
                    yield ("load", f"{nm}F{sl}", g // ns, {f"{nm}{sl}": f"{nm}({g})"})
                    last[f"{nm}F{sl}"] = g // ns
            for b in range(QB):
                used = [i for i in range(len(items)) if i % QB == b]
                if used:
                    yield ("wait", f"QDO{b}", used[-1] // QB)
            for bar, ph in last.items():
                yield ("wait", bar, ph)

        def gate():
            for g in range(G):
                if g + 1 < G:
                    yield ("wait", f"KF{(g + 1) % KS}", (g + 1) // KS)
                if g > 0:
                    yield ("wait", "LD", g - 1)
                yield ("arrive", "LD", 1, g)

        def copy_and_store():  # one warp: the item's dO copy, then its dQ store
            for it in range(len(items)):
                if copy_q:
                    yield ("wait", f"QDO{it % QB}", it // QB)
                    yield ("read", {f"dO{it % QB}": f"dO({it})"})
                    yield ("arrive", f"QE{it % QB}", 1, it // QB)
                yield ("wait", "EPF", it)
                yield ("read", every("ST", f"out({it})"))
                yield ("arrive", "EPE", 1, it)

        def s_mma(it, g):
            return ("mma", f"S({g})", dict(every(f"Q{it % QB}", f"Q({it})"), **{f"K{g % KS}": f"K({g})"}),
                    every("S", f"S({g})"))

        def dp_mma(it, g):
            return ("mma", f"dP({g})", {f"dO{it % QB}": f"dO({it})", f"V{g % VS}": f"V({g})"},
                    every(f"DP{g & 1}", f"dP({g})"))

        def dq_mma(it, j, g):
            reads = dict(every(f"DP{g & 1}", f"dS({g})"), **{f"K{g % KS}": f"K({g})"})
            if j > 0:
                reads["dQ"] = f"dQ({it},{j - 1})"
            return ("mma", f"dQ({g})", reads, {"dQ": f"dQ({it},{j})"})

        def mma():
            for it, nj in enumerate(items):
                g0 = starts[it]
                yield ("wait", f"QDO{it % QB}", it // QB)
                if it > 0 and mistake != "no_ld_cross":
                    yield ("wait", "LD", g0 - 1)  # S of the previous item's last block is read
                yield ("wait", f"KF{g0 % KS}", g0 // KS)
                yield s_mma(it, g0)
                yield ("wait", f"VF{g0 % VS}", g0 // VS)
                yield dp_mma(it, g0)
                yield ("commit", f"VE{g0 % VS}", g0 // VS)
                yield ("commit", "SDF", g0)
                if nj == 1:
                    yield ("commit", f"QE{it % QB}", it // QB)
                if nj > 1:
                    yield ("wait", f"VF{(g0 + 1) % VS}", (g0 + 1) // VS)
                    yield dp_mma(it, g0 + 1)
                    yield ("commit", f"VE{(g0 + 1) % VS}", (g0 + 1) // VS)
                for j in range(nj):
                    g = g0 + j
                    if j + 1 < nj:
                        yield ("wait", "LD", g)
                        yield ("wait", f"KF{(g + 1) % KS}", (g + 1) // KS)
                        yield s_mma(it, g + 1)
                        yield ("commit", "SDF", g + 1)
                        if j + 1 == nj - 1:
                            yield ("commit", f"QE{it % QB}", it // QB)  # the item's last S, dP issued
                    yield ("wait", "PF", g)
                    yield ("arrive", "PFS", 1, g)
                    yield dq_mma(it, j, g)
                    if j + 2 < nj:
                        yield ("wait", f"VF{(g + 2) % VS}", (g + 2) // VS)
                        yield dp_mma(it, g + 2)
                        yield ("commit", f"VE{(g + 2) % VS}", (g + 2) // VS)
                    yield ("commit", f"KE{g % KS}", g // KS)
                yield ("commit", "ACC", it)
            yield ("commit", "DONE", 0)
            yield ("wait", "DONE", 0)

        def compute(w, q):
            me = f"{w}.{q}"
            for it, nj in enumerate(items):
                for j in range(nj):
                    g = starts[it] + j
                    yield ("wait", "SDF", g)
                    yield ("read", {f"S.{me}": f"S({g})", f"DP{g & 1}.{me}": f"dP({g})"})
                    yield ("arrive", "LD", 32, g)
                    yield ("write", {f"DP{g & 1}.{me}": f"dS({g})"})
                    if g > 0:
                        yield ("wait", "PFS", g - 1)
                    yield ("arrive", "PF", 32, g)
                yield ("wait", "ACC", it)
                yield ("read", {"dQ": f"dQ({it},{nj - 1})"})
                if it > 0 and mistake != "no_epe":
                    yield ("wait", "EPE", it - 1)
                yield ("write", {f"ST.{me}": f"out({it})"})
                yield ("arrive", "EPF", 32, it)

        roles = {"prod": producer(), "gate": gate(), "mma": mma(), "copy": copy_and_store()}
        for w, q in warps:
            roles[f"c{w}{q}"] = compute(w, q)
        return bars, roles

    return model


def fwd_model(nkv0, nkv, NSLOT=4, copy_q=True, early_qk=False):
    """One CTA per work item with two query tiles, the epilogue staging O in
    the Q buffers behind a bar.sync (the forward kernels' earlier one-item
    form; both now run fwd_persistent_model's protocol, the FP8 forward as
    its d = 128 dense case without a copy warp): tile 0 multiplies key blocks [0, nkv0), tile 1
    [0, nkv) (nkv0 < nkv on the causal diagonal); four softmax warps per
    tile, warp q owning rows 32q.. of S_t and O_t; the epilogue stages O in
    Q_t's buffer."""
    rows = range(4)

    def model(rnd):
        bars = {"Q": 1, "SF0": 1, "SF1": 1, "PF0": 129, "PF1": 129, "OF0": 1, "OF1": 1,
                "DONE": 1, "QC": 1, "G1": 1}
        bars.update(ring_bars(NSLOT))
        n_of = (nkv0, nkv)

        def tile(pre, t, tag):
            return {f"{pre}.{t}.{q}": tag for q in rows}

        def gate():
            # the gate alone waits on the ring's full barriers, every entry in
            # order (K_0 too, passed on to the MMA thread on G1): a slot's
            # parity wait answers right only at the awaited phase or the one
            # after, and no slot can move on before the gate has let its entry
            # be used
            yield ("wait", "F0", 0)
            yield ("arrive", "G1", 1, 0)
            for j in range(nkv):
                v, kn = 2 * j + 1, 2 * j + 2
                yield ("wait", f"F{v % NSLOT}", v // NSLOT)
                if j + 1 < nkv:
                    yield ("wait", f"F{kn % NSLOT}", kn // NSLOT)
                for t in (0, 1):
                    if j >= n_of[t]:
                        continue
                    if j > 0:
                        yield ("wait", f"PF{t}", j - 1)
                    yield ("arrive", f"PF{t}", 1, j)

        def copy():
            yield ("wait", "Q", 0)
            yield ("read", dict(tile("Q", 0, "Q"), **tile("Q", 1, "Q")))
            yield ("arrive", "QC", 1, 0)

        def qk(t, j):
            slot = (2 * j) % NSLOT
            return ("mma", f"QK({t},{j})", dict(tile("Q", t, "Q"), **{f"kv{slot}": f"K({j})"}),
                    tile("S", t, f"S({t},{j})"))

        def pv(t, j):
            slot = (2 * j + 1) % NSLOT
            reads = dict(tile("S", t, f"P({t},{j})"), **{f"kv{slot}": f"V({j})"})
            if j > 0:
                reads.update(tile("O", t, f"O({t},{j - 1})"))
            return ("mma", f"PV({t},{j})", reads, tile("O", t, f"O({t},{j})"))

        def mma():
            yield ("wait", "Q", 0)
            yield ("wait", "G1", 0)
            yield qk(0, 0)
            yield ("commit", "SF0", 0)
            yield qk(1, 0)
            yield ("commit", "SF1", 0)
            yield ("commit", "E0", 0)
            for j in range(nkv):
                vslot, kidx = (2 * j + 1) % NSLOT, 2 * (j + 1)
                kslot = kidx % NSLOT
                if j < nkv0:
                    yield ("wait", "PF0", j)
                    yield pv(0, j)
                    if j == nkv0 - 1:
                        yield ("commit", "OF0", 0)
                if j + 1 < nkv0:
                    yield qk(0, j + 1)
                    yield ("commit", "SF0", j + 1)
                if early_qk and j + 1 < nkv:
                    yield qk(1, j + 1)
                yield ("wait", "PF1", j)
                yield pv(1, j)
                yield ("commit", f"E{vslot}", (2 * j + 1) // NSLOT)
                if j == nkv - 1:
                    yield ("commit", "OF1", 0)
                if j + 1 < nkv:
                    if not early_qk:
                        yield qk(1, j + 1)
                    yield ("commit", "SF1", j + 1)
                    yield ("commit", f"E{kslot}", kidx // NSLOT)
            yield ("commit", "DONE", 0)
            yield ("wait", "DONE", 0)

        def softmax(t, q):
            me = f"{t}.{q}"
            for j in range(n_of[t]):
                yield ("wait", f"SF{t}", j)
                yield ("read", {f"S.{me}": f"S({t},{j})"})
                yield ("write", {f"S.{me}": f"P({t},{j})"})
                if j > 0 and rnd.random() < 0.5:  # the reference max moved
                    yield ("read", {f"O.{me}": f"O({t},{j - 1})"})
                    yield ("write", {f"O.{me}": f"O({t},{j - 1})"})
                yield ("arrive", f"PF{t}", 32, j)
            yield ("wait", f"OF{t}", 0)
            if copy_q:
                yield ("wait", "QC", 0)
            yield ("read", {f"O.{me}": f"O({t},{n_of[t] - 1})"})
            yield ("write", {f"Q.{me}": "O tile"})  # staging in Q_t's buffer

        q_tiles = dict(tile("Q", 0, "Q"), **tile("Q", 1, "Q"))
        roles = {"prod": kv_ring_producer(nkv, NSLOT, q_tiles), "gate": gate(), "mma": mma()}
        for t in (0, 1):
            for q in rows:
                roles[f"s{t}{q}"] = softmax(t, q)
        if copy_q:
            roles["copy"] = copy()
        return bars, roles

    return model


def stream_entries(sets):
    """Ring order of the block-sparse forward: K_0(0), K_1(0), then per step k,
    tile by tile, V_t(k) and K_t(k+1) of the tiles that still have blocks (a
    tile's k-th block is the k-th of its own set)."""
    cnt = [len(sets[0]), len(sets[1])]
    seq = [(t, "K", 0) for t in (0, 1) if cnt[t] > 0]
    for k in range(max(cnt)):
        for t in (0, 1):
            if k < cnt[t]:
                seq.append((t, "V", k))
                if k + 1 < cnt[t]:
                    seq.append((t, "K", k + 1))
    return {e: i for i, e in enumerate(seq)}


def fwd_persistent_model(items, NSLOT=4, split_p=False, sparse=False, copy_q=False,
                         mistake=None, timeouts=False, drop=None, stage_q=False, epi_tma=False):
    """The persistent forward: one CTA walks `items`, each a pair (tile 0's key
    blocks, tile 1's key blocks).  Dense items (sparse=False) share K and V
    between the tiles, ring entries K(u), V(u) per block of tile 1's range;
    sparse items stream each tile's own blocks (stream_entries order).  The
    ring, the barrier phases and the tensor-core queues run on across items.
    O goes from TMEM straight to global memory, so the Q buffers are free for
    the next item once its score products and the copy warp are done with
    them (q_empty: one commit per issuer, one arrival from the copy warp).

    split_p (d = 64): P_t has columns of its own, and each tile has its own
    MMA issuer: S_t(k+1) as soon as s_empty(t) and K_t(k+1) allow (so also
    the first product of the next item), PV_t(k) on p_full(t) once V_t(k) has
    landed, committed to pv_done(t).  Dense rings are then released by both
    issuers (kv_empty counts 2); tile 0's issuer releases the entries of the
    blocks past its causal limit with plain arrivals once the slot's previous
    phase has completed.  Otherwise (d = 128, and the FP8 forward: dense,
    copy_q=False) one issuer, P over S_t, and a gate warp folding V(k),
    K(k+1) landed into p_full(t).

    timeouts: every wait is bounded (simulate_with_timeouts decides its
    outcome) and each role takes the kernel's failure path: it stops issuing,
    drains its own loads / MMAs, and meets the others at the teardown
    __syncthreads.  drop = (t, n): the n-th arrival for tile t that a partner
    owes (the gate's on p_full at d = 128, the softmax warps' on s_empty at
    d = 64) never happens.

    stage_q (the block-sparse kernel: one item per CTA): each tile's epilogue
    writes its O rows into the tile's own Q buffer, arrives on epi(t) (four
    warps), and the tile's first warp waits for it and stores the buffer (a
    TMA store, read here as a read of the four rows).  The buffer is free once
    o_final(t) has completed; a tile with no block waits for the Q load
    instead.

    epi_tma (a form of the dense kernel at d = 64 that was measured and not
    kept): each tile's epilogue writes its O rows into a staging buffer of
    the tile's own once the copy warp's stores of the previous item have read
    it (epi_empty(t)), and arrives on epi(t) (128 threads); the copy warp,
    after its Q copy, waits for epi(t), stores the buffer (a read of the four
    warps' rows) and arrives on epi_empty(t).

    mistake: "no_q_empty" (Q reloaded without q_empty), "early_arrive" (tile
    0's issuer arrives on kv_empty without the previous-phase wait),
    "no_k_wait" (a score product before its K tile has landed), "no_pvd_wait"
    (P_t written before the previous P V product has read it), "no_of_wait"
    (the epilogue reads O without o_final), "no_epe" (epi_tma: the staging
    rewritten without epi_empty), "no_drain" (the producer exits
    without waiting for its last loads), "mma_waits_first_k" (the issuer waits
    the item's first K entries itself and the gate starts at V(0): the gate's
    parity wait on a slot can then come a phase early or two late),
    "no_q_wait_empty" (stage_q: a tile with
    no block stages O without waiting for its Q load).  (The s_empty wait before an item's
    first score product is implied by q_empty: the issuer's commit to it
    follows its last P V product, which followed the softmax's p_full; the
    kernel keeps the wait anyway.)"""
    rows = range(4)
    items = [(sorted(set(a)), sorted(set(b))) for a, b in items]
    assert not stage_q or (sparse and len(items) == 1)
    nissue = 2 if split_p else 1
    n_roles = 1 + nissue + (0 if split_p else 1) + 8 + (1 if (copy_q or epi_tma) else 0)

    def entries(it):
        """the item's ring entries in order: (owner, kind, k) with owner a
        tile, or "both" for a dense entry (k is then the block)"""
        b0, b1 = it
        if not sparse:
            assert b0 == list(range(len(b0))) and b1 == list(range(len(b1)))
            assert len(b0) <= len(b1)
            return [e for u in range(len(b1)) for e in (("both", "K", u), ("both", "V", u))]
        return [e for e, _ in sorted(stream_entries(it).items(), key=lambda x: x[1])]

    ent, base = {}, 0
    for i, it in enumerate(items):
        seq = entries(it)
        for j, e in enumerate(seq):
            ent[(i,) + e] = base + j
        base += len(seq)

    def W(bar, phase, mode="abort"):
        return ("twait", bar, phase, mode) if timeouts else ("wait", bar, phase)

    def model(rnd):
        bars = {"Q": 1, "QE": nissue + (1 if copy_q else 0), "DONE": nissue, "G1": 1}
        for t in (0, 1):
            bars.update({f"SF{t}": 1, f"PF{t}": 128 if split_p else 129, f"OF{t}": 1,
                         f"SE{t}": 4, f"PVD{t}": 1, f"EPI{t}": 128 if epi_tma else 4,
                         f"EPE{t}": 1})
        for s in range(NSLOT):
            bars[f"F{s}"] = 1
            bars[f"E{s}"] = 2 if (split_p and not sparse) else 1

        def tile(pre, t, tag):
            return {f"{pre}.{t}.{q}": tag for q in rows}

        def teardown():
            if timeouts:
                yield ("nbar", "syncthreads", n_roles)

        def slot(i, t, w, k):
            e = ent[(i, "both" if not sparse else t, w, items[i][t][k] if not sparse else k)]
            return e % NSLOT, e // NSLOT

        def kv_tag(i, t, w, k):
            return f"{w}{'' if not sparse else t}({i},{items[i][t][k]})"

        def producer():
            last, ok, nq = {}, True, 0
            for i, it in enumerate(items):
                if i > 0 and mistake != "no_q_empty":
                    ok = (yield W("QE", i - 1)) is not False
                    if not ok:
                        break
                yield ("load", "Q", i, dict(tile("Q", 0, f"Q{i}"), **tile("Q", 1, f"Q{i}")))
                nq = i + 1
                for e in entries(it):
                    owner, w, k = e
                    g = ent[(i,) + e]
                    s = g % NSLOT
                    ok = (yield W(f"E{s}", g // NSLOT - 1)) is not False
                    if not ok:
                        break
                    tag = f"{w}({i},{k})" if owner == "both" else f"{w}{owner}({i},{it[owner][k]})"
                    yield ("load", f"F{s}", g // NSLOT, {f"kv{s}": tag})
                    last[s] = g // NSLOT
                if not ok:
                    break
            if mistake != "no_drain":
                if nq:
                    yield W("Q", nq - 1, "drain")
                for s, ph in last.items():
                    yield W(f"F{s}", ph, "drain")
            yield from teardown()

        def qk(i, t, k):
            s, _ = slot(i, t, "K", k)
            return ("mma", f"QK{t}({i},{k})", dict(tile("Q", t, f"Q{i}"), **{f"kv{s}": kv_tag(i, t, "K", k)}),
                    tile("S", t, f"S{t}({i},{k})"))

        def pv(i, t, k):
            s, _ = slot(i, t, "V", k)
            reads = dict(tile("P" if split_p else "S", t, f"P{t}({i},{k})"),
                         **{f"kv{s}": kv_tag(i, t, "V", k)})
            if k > 0:
                reads.update(tile("O", t, f"O{t}({i},{k - 1})"))
            return ("mma", f"PV{t}({i},{k})", reads, tile("O", t, f"O{t}({i},{k})"))

        def release(i, t, w, k):
            s, ph = slot(i, t, w, k)
            return ("commit", f"E{s}", ph)

        def gate():  # d = 128: V(k), K(k+1) landed -> p_full(t)
            pf, ok, ng1 = [0, 0], True, 0
            for i, it in enumerate(items):
                # the item's first K entries too, so that the gate sees every
                # ring phase in order (a slot's parity wait answers right only
                # once the phase before it was seen done)
                firsts = [(1, "K", 0)] if not sparse and it[1] else \
                    [(t, "K", 0) for t in (0, 1) if sparse and it[t]]
                if mistake == "mma_waits_first_k":
                    firsts = []
                for (tt, w, kk) in firsts:
                    s, ph = slot(i, tt, w, kk)
                    if ok:
                        ok = (yield W(f"F{s}", ph)) is not False
                if not ok:
                    break
                if firsts:  # the MMA thread's first score products wait on this
                    yield ("arrive", "G1", 1, ng1)
                    ng1 += 1
                if not sparse:
                    steps = [(u, [t for t in (0, 1) if u < len(it[t])]) for u in range(len(it[1]))]
                else:
                    steps = [(k, [t for t in (0, 1) if k < len(it[t])])
                             for k in range(max(len(it[0]), len(it[1]), 0))]
                for k, tiles in steps:
                    waits = []  # (tile, kind, k) of the entries that must have landed
                    if not sparse:  # dense: one pair serves both tiles
                        waits = [(1, "V", k)] + ([(1, "K", k + 1)] if k + 1 < len(it[1]) else [])
                    for t in tiles:
                        if sparse:
                            waits = [(t, "V", k)] + ([(t, "K", k + 1)] if k + 1 < len(it[t]) else [])
                        for (tt, w, kk) in waits:
                            s, ph = slot(i, tt, w, kk)
                            if ok:
                                ok = (yield W(f"F{s}", ph)) is not False
                        waits = []
                        if ok and pf[t] > 0:
                            ok = (yield W(f"PF{t}", pf[t] - 1)) is not False
                        if not ok:
                            break
                        if (t, pf[t]) != drop:
                            yield ("arrive", f"PF{t}", 1, pf[t])
                        pf[t] += 1
                    if not ok:
                        break
                if not ok:
                    break
            yield from teardown()

        def issuer_split(t):
            nqk = npv = nof = 0
            ok = True
            for i, it in enumerate(items):
                ok = (yield W("Q", i)) is not False
                if not ok:
                    break
                bl = it[t]
                for k in range(len(bl) + 1):
                    if k < len(bl):  # S_t(k) (k = 0: the item's first)
                        if nqk > 0:
                            ok = (yield W(f"SE{t}", nqk - 1)) is not False
                        s, ph = slot(i, t, "K", k)
                        if ok and mistake != "no_k_wait":
                            ok = (yield W(f"F{s}", ph)) is not False
                        if not ok:
                            break
                        yield qk(i, t, k)
                        yield ("commit", f"SF{t}", nqk)
                        yield release(i, t, "K", k)
                        nqk += 1
                    if k > 0:  # PV_t(k - 1)
                        s, ph = slot(i, t, "V", k - 1)
                        ok = (yield W(f"F{s}", ph)) is not False
                        if ok:
                            ok = (yield W(f"PF{t}", npv)) is not False
                        if not ok:
                            break
                        yield pv(i, t, k - 1)
                        yield ("commit", f"PVD{t}", npv)
                        yield release(i, t, "V", k - 1)
                        npv += 1
                        if k == len(bl):
                            yield ("commit", f"OF{t}", nof)
                            nof += 1
                if ok and not sparse and t == 0:  # blocks past tile 0's limit
                    for u in range(len(it[0]), len(it[1])):
                        for w in ("K", "V"):
                            s, ph = slot(i, 1, w, u)
                            if mistake != "early_arrive":
                                ok = (yield W(f"E{s}", ph - 1)) is not False
                            if not ok:
                                break
                            yield ("arrive", f"E{s}", 1, ph)
                        if not ok:
                            break
                if not ok:
                    break
                yield ("commit", "QE", i)
            yield ("commit", "DONE", 0)
            if t == 0:
                yield W("DONE", 0, "drain")
            yield from teardown()

        def issuer_single():
            npv, nof, nsf = [0, 0], [0, 0], [0, 0]
            ok, ng1 = True, 0
            for i, it in enumerate(items):
                ok = (yield W("Q", i)) is not False
                if ok and (it[0] or it[1]) and mistake != "mma_waits_first_k":
                    # the gate has seen the item's first K entries
                    ok = (yield W("G1", ng1)) is not False
                    ng1 += 1
                for t in (0, 1):
                    if not ok:
                        break
                    if it[t] and mistake == "mma_waits_first_k" and (sparse or t == 0):
                        s, ph = slot(i, t, "K", 0)
                        ok = (yield W(f"F{s}", ph)) is not False
                        if not ok:
                            break
                    if it[t]:
                        yield qk(i, t, 0)
                        yield ("commit", f"SF{t}", nsf[t])
                        nsf[t] += 1
                        if sparse or t == 1:
                            yield release(i, t, "K", 0)
                steps = len(it[1]) if not sparse else max(len(it[0]), len(it[1]), 0)
                for k in range(steps):
                    for t in (0, 1):
                        if not ok or k >= len(it[t]):
                            continue
                        ok = (yield W(f"PF{t}", npv[t])) is not False
                        if not ok:
                            break
                        yield pv(i, t, k)
                        npv[t] += 1
                        if sparse or t == 1:
                            yield release(i, t, "V", k)
                        if k == len(it[t]) - 1:
                            yield ("commit", f"OF{t}", nof[t])
                            nof[t] += 1
                        if k + 1 < len(it[t]):
                            yield qk(i, t, k + 1)
                            yield ("commit", f"SF{t}", nsf[t])
                            nsf[t] += 1
                            if sparse or t == 1:
                                yield release(i, t, "K", k + 1)
                    if not ok:
                        break
                if not ok:
                    break
                yield ("commit", "QE", i)
            yield ("commit", "DONE", 0)
            yield W("DONE", 0, "drain")
            yield from teardown()

        def copy():
            ok = True
            for i in range(len(items)):
                if copy_q:
                    ok = (yield W("Q", i)) is not False
                    if not ok:
                        break
                    yield ("read", dict(tile("Q", 0, f"Q{i}"), **tile("Q", 1, f"Q{i}")))
                    yield ("arrive", "QE", 1, i)
                if epi_tma:
                    for t in (0, 1):
                        ok = (yield W(f"EPI{t}", i)) is not False
                        if not ok:
                            break
                        yield ("read", {f"ST.{t}.{qq}": f"Ostage{t}({i})" for qq in rows})
                        yield ("arrive", f"EPE{t}", 1, i)
                    if not ok:
                        break
            yield from teardown()

        def softmax(t, q):
            me = f"{t}.{q}"
            nsf = npv = nof = 0
            ok = True
            for i, it in enumerate(items):
                bl = it[t]
                for k in range(len(bl)):
                    ok = (yield W(f"SF{t}", nsf)) is not False
                    if not ok:
                        break
                    nsf += 1
                    yield ("read", {f"S.{me}": f"S{t}({i},{k})"})
                    if split_p:
                        if (t, nsf - 1) != drop:
                            yield ("arrive", f"SE{t}", 1, nsf - 1)
                        if k > 0 and mistake != "no_pvd_wait":
                            ok = (yield W(f"PVD{t}", npv - 1)) is not False
                            if not ok:
                                break
                        yield ("write", {f"P.{me}": f"P{t}({i},{k})"})
                    else:
                        yield ("write", {f"S.{me}": f"P{t}({i},{k})"})
                    if k > 0 and rnd.random() < 0.5:  # the reference max moved
                        yield ("read", {f"O.{me}": f"O{t}({i},{k - 1})"})
                        yield ("write", {f"O.{me}": f"O{t}({i},{k - 1})"})
                    yield ("arrive", f"PF{t}", 32, npv)
                    npv += 1
                if not ok:
                    break
                if bl:
                    if mistake != "no_of_wait":
                        ok = (yield W(f"OF{t}", nof)) is not False
                        if not ok:
                            break
                    nof += 1
                    yield ("read", {f"O.{me}": f"O{t}({i},{len(bl) - 1})"})
                elif stage_q and mistake != "no_q_wait_empty":
                    ok = (yield W("Q", i)) is not False
                    if not ok:
                        break
                if epi_tma:
                    if i > 0 and mistake != "no_epe":
                        ok = (yield W(f"EPE{t}", i - 1)) is not False
                        if not ok:
                            break
                    yield ("write", {f"ST.{me}": f"Ostage{t}({i})"})
                    yield ("arrive", f"EPI{t}", 32, i)
                if stage_q:
                    yield ("write", {f"Q.{me}": f"Ostage{t}"})
                    yield ("arrive", f"EPI{t}", 1, 0)
                    if q == 0:
                        ok = (yield W(f"EPI{t}", 0)) is not False
                        if not ok:
                            break
                        yield ("read", {f"Q.{t}.{qq}": f"Ostage{t}" for qq in rows})
            yield from teardown()

        roles = {"prod": producer()}
        if split_p:
            roles["mma0"], roles["mma1"] = issuer_split(0), issuer_split(1)
        else:
            roles["mma"], roles["gate"] = issuer_single(), gate()
        for t in (0, 1):
            for q in rows:
                roles[f"s{t}{q}"] = softmax(t, q)
        if copy_q or epi_tma:
            roles["copy"] = copy()
        return bars, roles

    return model


# ----------------------------------------------- split-KV (decode) kernel
def decode_model(nkv, NSLOT=6, skip_pvd_wait=False):
    """Four softmax warps, warp q owning rows 32q.. of S0, S1 and O."""
    rows = range(4)

    def model(rnd):
        bars = {"Q": 1, "SF0": 1, "SF1": 1, "PF0": 128, "PF1": 128, "PVD": 1, "OF": 1}
        bars.update(ring_bars(NSLOT))

        def every(pre, tag):
            return {f"{pre}.{q}": tag for q in rows}

        def landed(idx):
            return ("wait", f"F{idx % NSLOT}", idx // NSLOT)

        def issue_s(j):
            idx = 2 * j
            yield landed(idx)
            yield ("mma", f"S({j})", {"Q": "Q", f"kv{idx % NSLOT}": f"K({j})"},
                   every(f"S{j & 1}", f"S({j})"))
            yield ("commit", f"SF{j & 1}", j >> 1)
            yield ("commit", f"E{idx % NSLOT}", idx // NSLOT)

        def mma():
            if nkv == 0:
                return
            yield ("wait", "Q", 0)
            yield from issue_s(0)
            for j in range(nkv):
                if j + 1 < nkv:
                    yield from issue_s(j + 1)
                yield ("wait", f"PF{j & 1}", j >> 1)
                idx = 2 * j + 1
                yield landed(idx)
                reads = dict(every(f"S{j & 1}", f"P({j})"), **{f"kv{idx % NSLOT}": f"V({j})"})
                if j > 0:
                    reads.update(every("O", f"O({j - 1})"))
                yield ("mma", f"PV({j})", reads, every("O", f"O({j})"))
                yield ("commit", f"E{idx % NSLOT}", idx // NSLOT)
                yield ("commit", "PVD", j)
            yield ("commit", "OF", 0)
            yield ("wait", "OF", 0)

        def softmax(q):
            for j in range(nkv):
                yield ("wait", f"SF{j & 1}", j >> 1)
                yield ("read", {f"S{j & 1}.{q}": f"S({j})"})
                yield ("write", {f"S{j & 1}.{q}": f"P({j})"})
                if j > 0 and rnd.random() < 0.5:  # the reference max moved
                    if not skip_pvd_wait:
                        yield ("wait", "PVD", j - 1)
                    yield ("read", {f"O.{q}": f"O({j - 1})"})
                    yield ("write", {f"O.{q}": f"O({j - 1})"})
                yield ("arrive", f"PF{j & 1}", 32, j >> 1)
            if nkv > 0:
                yield ("wait", "OF", 0)
                yield ("read", {f"O.{q}": f"O({nkv - 1})"})

        roles = {"prod": kv_ring_producer(nkv, NSLOT, {"Q": "Q"}), "mma": mma()}
        for q in rows:
            roles[f"s{q}"] = softmax(q)
        return bars, roles

    return model


# ---------------------- single S buffer (one-tile forward; no kernel uses it now)
# The FP8 forward now has the bf16 forward's two-tile protocol (fwd_model with
# no copy warp, which test_forward_protocol runs).  This model of the earlier
# one-tile protocol stays as the ring-without-empty-wait planted-mistake case.
def single_s_model(nkv, NSLOT=4, skip_empty=False):
    """Four softmax warps over one S buffer (P written over S), a ring of
    NSLOT K / V^T tiles."""
    rows = range(4)

    def model(rnd):
        bars = {"Q": 1, "SF": 1, "PF": 128, "OF": 1}
        bars.update(ring_bars(NSLOT))

        def every(pre, tag):
            return {f"{pre}.{q}": tag for q in rows}

        def landed(idx):
            return ("wait", f"F{idx % NSLOT}", idx // NSLOT)

        def issue_s(j):
            idx = 2 * j
            yield landed(idx)
            yield ("mma", f"S({j})", {"Q": "Q", f"kv{idx % NSLOT}": f"K({j})"},
                   every("S", f"S({j})"))
            yield ("commit", "SF", j)
            yield ("commit", f"E{idx % NSLOT}", idx // NSLOT)

        def mma():
            yield ("wait", "Q", 0)
            yield from issue_s(0)
            for j in range(nkv):
                yield ("wait", "PF", j)
                idx = 2 * j + 1
                yield landed(idx)
                reads = dict(every("S", f"P({j})"), **{f"kv{idx % NSLOT}": f"V^T({j})"})
                if j > 0:
                    reads.update(every("O", f"O({j - 1})"))
                yield ("mma", f"PV({j})", reads, every("O", f"O({j})"))
                yield ("commit", f"E{idx % NSLOT}", idx // NSLOT)
                if j + 1 < nkv:
                    yield from issue_s(j + 1)
            yield ("commit", "OF", 0)
            yield ("wait", "OF", 0)

        def softmax(q):
            for j in range(nkv):
                yield ("wait", "SF", j)
                yield ("read", {f"S.{q}": f"S({j})"})
                yield ("write", {f"S.{q}": f"P({j})"})
                if j > 0 and rnd.random() < 0.5:
                    yield ("read", {f"O.{q}": f"O({j - 1})"})
                    yield ("write", {f"O.{q}": f"O({j - 1})"})
                yield ("arrive", "PF", 32, j)
            yield ("wait", "OF", 0)
            yield ("read", {f"O.{q}": f"O({nkv - 1})"})

        prod = kv_ring_producer(nkv, NSLOT, {"Q": "Q"}, tiles=("K", "V^T"), skip_empty=skip_empty)
        roles = {"prod": prod, "mma": mma()}
        for q in rows:
            roles[f"s{q}"] = softmax(q)
        return bars, roles

    return model


# ------------------------------------------------------------------ the kernels
@pytest.mark.parametrize("nj", [1, 2, 3, 4, 7, 20])
@pytest.mark.parametrize("two_issuers,early_dp", [(False, False), (True, False), (False, True)])
def test_dq_protocol(nj, two_issuers, early_dp):
    each_seed(dq_model(nj, two_issuers=two_issuers, early_dp=early_dp))


@pytest.mark.parametrize("nj", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("ks,vs", [(3, 2), (4, 3)])
def test_dq_protocol_late_ke(nj, ks, vs):
    each_seed(dq_model(nj, KS=ks, VS=vs, early_dp=True, late_ke=True))


@pytest.mark.parametrize("nj", [1, 2, 3, 5, 16])
def test_dq_protocol_deep_rings(nj):
    # d = 64: four K and three V ring slots
    each_seed(dq_model(nj, KS=4, VS=3, early_dp=True))


DKDV_PERSISTENT_ITEMS = [[1], [2], [3], [16, 16], [1, 1, 1], [2, 3, 1, 4], [5, 1, 2], [3] * 6]


@pytest.mark.parametrize("items", range(len(DKDV_PERSISTENT_ITEMS)))
@pytest.mark.parametrize("lagging_store", [False, True])
@pytest.mark.parametrize("kvb", [1, 2])
def test_dkdv_persistent_protocol(items, lagging_store, kvb):
    each_seed(dkdv_persistent_model(DKDV_PERSISTENT_ITEMS[items], lagging_store=lagging_store,
                                    kv_buffers=kvb),
              seeds=range(40))


@pytest.mark.parametrize("mistake,items,lag,kvb", [("no_kve", [3, 2, 4], False, 1),
                                                   ("no_kve", [1, 1, 2, 1, 3], False, 2),
                                                   ("no_epe", [2, 1, 3], True, 1),
                                                   ("no_epe", [2, 1, 3], True, 2)])
def test_dkdv_persistent_planted_mistakes_are_caught(mistake, items, lag, kvb):
    assert fails_on_some_seed(dkdv_persistent_model(items, mistake=mistake, lagging_store=lag,
                                                    kv_buffers=kvb),
                              seeds=range(200))


DQ_PERSISTENT_ITEMS = [[1], [2], [3], [16, 16], [1, 1, 1], [2, 3, 1, 4], [5, 1, 2], [3] * 6]


@pytest.mark.parametrize("items", range(len(DQ_PERSISTENT_ITEMS)))
@pytest.mark.parametrize("copy_q", [False, True])
@pytest.mark.parametrize("qb", [1, 2])
def test_dq_persistent_protocol(items, copy_q, qb):
    each_seed(dq_persistent_model(DQ_PERSISTENT_ITEMS[items], copy_q=copy_q, qdo_buffers=qb),
              seeds=range(40))


@pytest.mark.parametrize("mistake,items,qb,nseeds", [("no_qe", [3, 2, 4], 1, 200),
                                                     ("no_qe", [1, 1, 2, 1, 3], 2, 200),
                                                     ("no_ld_cross", [3, 2, 4], 1, 200),
                                                     ("no_ld_cross", [4, 1, 1, 4], 2, 400),
                                                     ("no_epe", [1] * 6, 1, 200),
                                                     ("no_epe", [1] * 6, 2, 200)])
def test_dq_persistent_planted_mistakes_are_caught(mistake, items, qb, nseeds):
    # (a store thread a whole item late needs short items to show; with two
    # Q/dO buffers the LD parity alias needs a one-block item between longer
    # ones and shows on few schedules)
    assert fails_on_some_seed(dq_persistent_model(items, mistake=mistake, qdo_buffers=qb),
                              seeds=range(nseeds))


def test_dq_early_dp_before_dq_is_caught():
    # dP(j+2) issued before dQ(j): it overwrites dS(j) before dQ(j) reads it
    assert fails_on_some_seed(dq_model(6, early_dp=True, dp_before_dq=True))


@pytest.mark.parametrize("n_it", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("three_regions", [False, True])
def test_dkdv_protocol(n_it, three_regions):
    each_seed(dkdv_model(n_it, three_regions=three_regions))


@pytest.mark.parametrize("n_it", [1, 3, 16])
@pytest.mark.parametrize("ds_in_do", [True, False])
def test_dkdv_smem_ds_variant_protocol(n_it, ds_in_do):
    each_seed(dkdv_model(n_it, ds_smem=True, ds_in_do=ds_in_do))


@pytest.mark.parametrize("nkv0,nkv,nslot", [(1, 1, 4), (1, 2, 4), (2, 3, 4), (5, 6, 4), (8, 8, 4),
                                            (3, 4, 8), (9, 9, 8)])
@pytest.mark.parametrize("copy_q", [True, False])
def test_forward_protocol(nkv0, nkv, nslot, copy_q):
    each_seed(fwd_model(nkv0, nkv, nslot, copy_q))


PERSISTENT_DENSE = [  # (tile 0's blocks, tile 1's blocks) per item: causal diagonal and full rows
    [(range(3), range(4)), (range(4), range(4)), (range(1), range(2)), (range(5), range(6))],
    [(range(1), range(1))] * 4,
    [(range(7), range(8)), (range(2), range(3))],
]
PERSISTENT_SPARSE = [
    [([0, 2, 3], [1, 2]), ([], [0, 3]), ([1], []), ([], []), ([0, 1, 2, 3], [0, 1, 2, 3])],
    [([0, 1, 5], [0, 4, 5, 6]), ([2], [2]), ([0, 3, 6], [1])],
]


@pytest.mark.parametrize("items", range(len(PERSISTENT_DENSE)))
@pytest.mark.parametrize("split_p,nslot", [(False, 4), (True, 8), (True, 4)])
@pytest.mark.parametrize("copy_q", [False, True])
def test_forward_persistent_dense_protocol(items, split_p, nslot, copy_q):
    each_seed(fwd_persistent_model(PERSISTENT_DENSE[items], nslot, split_p=split_p, copy_q=copy_q),
              seeds=range(40))


@pytest.mark.parametrize("items", range(len(PERSISTENT_DENSE)))
@pytest.mark.parametrize("copy_q", [False, True])
def test_forward_persistent_dense_staged_epilogue_protocol(items, copy_q):
    # d = 64 dense with O staged per tile for the copy warp's TMA stores (a
    # measured form, not kept)
    each_seed(fwd_persistent_model(PERSISTENT_DENSE[items], 8, split_p=True, copy_q=copy_q,
                                   epi_tma=True), seeds=range(40))


@pytest.mark.parametrize("copy_q", [False, True])
def test_forward_staging_rewritten_before_its_store_is_caught(copy_q):
    items = [([0], [0])] * 4  # short items, so a slow copy warp lags a whole item
    assert fails_on_some_seed(fwd_persistent_model(items, 8, split_p=True, copy_q=copy_q,
                                                   epi_tma=True, mistake="no_epe"),
                              seeds=range(300))


@pytest.mark.parametrize("items", range(len(PERSISTENT_SPARSE)))
@pytest.mark.parametrize("split_p,nslot", [(False, 5), (False, 4), (True, 8)])
def test_forward_persistent_sparse_protocol(items, split_p, nslot):
    each_seed(fwd_persistent_model(PERSISTENT_SPARSE[items], nslot, split_p=split_p, sparse=True),
              seeds=range(40))


SPARSE_ONE_ITEM = [it for case in PERSISTENT_SPARSE for it in case]


@pytest.mark.parametrize("item", range(len(SPARSE_ONE_ITEM)))
@pytest.mark.parametrize("split_p,nslot", [(False, 5), (True, 8)])
def test_forward_sparse_one_item_epilogue_in_q_buffer(item, split_p, nslot):
    # the block-sparse kernel: one item per CTA, O staged in the tile's own Q
    # buffer and stored from there
    each_seed(fwd_persistent_model([SPARSE_ONE_ITEM[item]], nslot, split_p=split_p, sparse=True,
                                   stage_q=True), seeds=range(60))


@pytest.mark.parametrize("split_p,nslot", [(False, 5), (True, 8)])
def test_forward_sparse_empty_tile_must_wait_for_its_q_load(split_p, nslot):
    # a tile with no block stages O over a Q load that may still be landing
    assert fails_on_some_seed(fwd_persistent_model([([], [0, 3])], nslot, split_p=split_p,
                                                   sparse=True, stage_q=True,
                                                   mistake="no_q_wait_empty"))


@pytest.mark.parametrize("sparse", [False, True])
def test_forward_gate_that_skips_first_k_is_caught(sparse):
    items = PERSISTENT_SPARSE[0] if sparse else PERSISTENT_DENSE[0]
    assert fails_on_some_seed(fwd_persistent_model(items, 5 if sparse else 4, sparse=sparse,
                                                   mistake="mma_waits_first_k"))


def test_forward_persistent_random_masks():
    rnd = random.Random(13)
    for _ in range(25):
        items = []
        for _ in range(rnd.randrange(1, 5)):
            nb = rnd.randrange(1, 9)
            items.append(([u for u in range(nb) if rnd.random() < 0.5],
                          [u for u in range(nb) if rnd.random() < 0.5]))
        split_p = rnd.random() < 0.5
        each_seed(fwd_persistent_model(items, 8 if split_p else rnd.choice((4, 5)), split_p=split_p,
                                       sparse=True), seeds=range(8))


@pytest.mark.parametrize("mistake,split_p", [("no_q_empty", False), ("no_q_empty", True),
                                             ("early_arrive", True), ("no_of_wait", False),
                                             ("no_of_wait", True), ("no_k_wait", True),
                                             ("no_pvd_wait", True)])
def test_forward_persistent_planted_mistakes_are_caught(mistake, split_p):
    assert fails_on_some_seed(fwd_persistent_model(PERSISTENT_DENSE[0], 8 if split_p else 4,
                                                   split_p=split_p, copy_q=True, mistake=mistake))


@pytest.mark.parametrize("nkv,nslot", [(0, 6), (1, 6), (2, 6), (3, 6), (7, 6), (20, 6), (13, 12)])
def test_decode_protocol(nkv, nslot):
    each_seed(decode_model(nkv, nslot))


@pytest.mark.parametrize("nkv", [1, 2, 3, 9])
def test_single_s_protocol(nkv):
    each_seed(single_s_model(nkv))


# ------------------------------------------------------- planted mistakes
def test_dq_first_gate_design_is_caught():
    assert fails_on_some_seed(dq_model(12, handshake=False, first_gate_design=True))


def test_dq_without_handshake_is_caught():
    # without it, a warp that runs a block ahead adds its dS(j) arrival to the
    # phase of dS(j-1), or dS(j+1) completes before the MMA thread has seen
    # dS(j), and its parity wait reads the phase as open
    assert fails_on_some_seed(dq_model(6, handshake=False))


def test_dq_two_issuers_without_dq_done_is_caught():
    # dP(j+2) written over dS(j) before the other thread's dQ(j) has read it
    assert fails_on_some_seed(dq_model(8, two_issuers=True, skip_dqd=True))


def test_dq_two_issuers_single_dq_done_barrier_is_caught():
    # one DQD barrier for both dP buffers: the dQ thread can complete two of
    # its phases before the S/dP thread waits, and the parity then aliases
    assert fails_on_some_seed(dq_model(8, two_issuers=True, single_dqd=True))


def test_forward_early_score_product_is_caught():
    # S(1, j+1) issued before the softmax has handed P(1, j) back
    assert fails_on_some_seed(fwd_model(3, 4, early_qk=True))


def test_decode_rescale_without_pv_wait_is_caught():
    # O rescaled while P(j-1) V_{j-1} may still be accumulating into it
    assert fails_on_some_seed(decode_model(12, skip_pvd_wait=True))


@pytest.mark.parametrize("n_it", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("nst", [2, 3])
def test_dkdv_protocol_late_ste(n_it, nst):
    each_seed(dkdv_model(n_it, NST=nst, late_ste=True))


@pytest.mark.parametrize("n_it", [1, 2, 4, 16])
def test_dkdv_protocol_three_stages(n_it):
    # d = 64: three {Q, dO} stages
    each_seed(dkdv_model(n_it, NST=3))


def test_dkdv_dk_before_ds_is_caught():
    # dK += dS^T Q issued before the warpgroups have written dS^T
    assert fails_on_some_seed(dkdv_model(4, dk_before_dsf=True))


def test_dkdv_p_before_s_ready_is_caught():
    # P^T formed from the region before S^T has been written there
    assert fails_on_some_seed(dkdv_model(4, p_before_str=True))


def test_dkdv_three_regions_without_dsf_handshake_is_caught():
    assert fails_on_some_seed(dkdv_model(5, three_regions=True, skip_dsf_wait=True))


def test_dkdv_early_dp_without_third_region_is_caught():
    # dP^T(it+1) issued before dK(it) with only two regions: it overwrites
    # P^T(it), dS^T(it) before dK(it) and the warps have used them
    assert fails_on_some_seed(dkdv_model(4, early_dpt=True))


@pytest.mark.parametrize("ds_in_do", [True, False])
def test_dkdv_ds_write_without_dv_done_is_caught(ds_in_do):
    # dS^T written over the dO tile before dV(it) has read it (d = 128), or
    # into its own buffer before dK(it-1) has read the previous one (d = 64)
    assert fails_on_some_seed(dkdv_model(5, ds_smem=True, ds_in_do=ds_in_do, skip_dvd=True))


def test_ring_without_empty_wait_is_caught():
    # a load into a ring slot whose previous tile an MMA still has to read
    assert fails_on_some_seed(single_s_model(9, skip_empty=True))


# ----------------------------------------------- the forward's time-out path
# The kernels bound every mbarrier wait.  A wait that runs out records the
# failure (status word) and returns false; a pending wait of the same launch
# that sees a recorded failure returns false within a few polls; the waits a
# block makes for its own copies and MMAs before it exits (mbar_drain) ignore
# other blocks' failures and give up on their time limit alone.  Every other
# wait in the kernels is either hardware-bounded (tcgen05.wait::ld/st, the TMA
# store's wait_group.read) or a bar.sync that every participating thread
# reaches on every path.  The model below runs the forward kernel's roles as
# generators that receive each bounded wait's result, exactly as the CUDA code
# branches on it, with named barriers (bar.sync) and the block-wide teardown
# barrier that block until every participant arrives.  Faults: waits that run
# out at random (any wait, any time), or an arrival that never happens.  In
# every schedule the block must reach its teardown (no bar.sync left waiting),
# with no load or MMA in flight, and with the failure recorded when a wait ran
# out.


def simulate_with_timeouts(model, seed, p_spurious=0.0, limit=400, max_steps=2000000,
                           p_load=None):
    rnd = random.Random(seed)
    bars, roles = model(random.Random(seed + 7))
    cta = Cta(bars)
    state = {"failed": False}
    speed = {r: rnd.choice((0.05, 0.3, 1.0)) for r in sorted(roles)}
    p_load0, p_tc = rnd.choice((0.05, 0.3, 1.0)), rnd.choice((0.05, 0.3, 1.0))
    p_load = p_load0 if p_load is None else p_load  # a fixed rate: slow copies
    cur, polls, nbar = {}, {}, {}

    def advance(r, value):
        try:
            cur[r] = op = roles[r].send(value)
        except StopIteration:
            del cur[r]
            return
        if op[0] == "nbar":  # a thread arrives at bar.sync as soon as it reaches it
            _, name, count = op
            waiting = nbar.setdefault(name, set())
            waiting.add(r)
            if len(waiting) == count:
                del nbar[name]
                if name == "syncthreads" and (cta.tc_busy() or cta.loads):
                    # the block exits (and frees its TMEM) right after this barrier
                    raise ProtocolError(f"teardown with work in flight: {cta.tcq} {cta.loads[:2]}")
                for w in sorted(waiting):
                    advance(w, None)

    for r in roles:
        advance(r, None)
    for _ in range(max_steps):
        if not cur:
            if cta.tc_busy() or cta.loads:
                raise ProtocolError(f"exit with work in flight: {cta.tcq} {cta.loads[:2]}")
            return state["failed"]
        progressed = False
        for r in rnd.sample(sorted(cur), len(cur)):
            if r not in cur or rnd.random() >= speed[r]:
                continue
            op = cur[r]
            if op[0] == "twait":
                _, bar, phase, mode = op
                try:
                    done = cta.bars[bar].done(phase)
                except ProtocolError as e:
                    raise ProtocolError(f"{r}: {e}") from None
                if done:
                    polls.pop(r, None)
                    advance(r, True)
                    progressed = True
                    continue
                polls[r] = polls.get(r, 0) + 1
                runs_out = polls[r] > (50 * limit if mode == "drain" else limit) or (
                    mode == "abort" and rnd.random() < p_spurious)
                gives_up = mode == "abort" and state["failed"] and polls[r] >= 16
                if runs_out or gives_up:
                    state["failed"] |= runs_out
                    polls.pop(r, None)
                    advance(r, False)
                    progressed = True
            elif op[0] == "nbar":
                continue  # released by the last participant's arrival
            else:
                cta.step(r, op)
                advance(r, None)
                progressed = True
        if cta.loads and rnd.random() < p_load:
            cta.land(rnd.randrange(len(cta.loads)))
            progressed = True
        if cta.tc_busy() and rnd.random() < p_tc:
            cta.run_tc(rnd)
            progressed = True
        if (not progressed and not cta.tc_busy() and not cta.loads and cur
                and all(op[0] == "nbar" for op in cur.values())):
            raise ProtocolError(f"bar.sync never completes: {nbar}")
    raise ProtocolError("did not finish")


def fwd_timeout_model(nkv0, nkv, NSLOT=4, copy_q=True, drop=None):
    """The one-item two-tile forward's roles (the earlier form of both
    forward kernels) with every bounded wait's two outcomes:
    producer, gate, copy warp, MMA thread and the eight softmax warps (four
    per query tile), the epilogue's bar.sync over a tile's four warps, and the
    teardown __syncthreads over every role.  drop = (t, j): the gate's
    arrival on p_full(t) for key block j never happens (a protocol fault)."""
    rows = range(4)

    def model(rnd):
        bars = {"Q": 1, "SF0": 1, "SF1": 1, "PF0": 129, "PF1": 129, "OF0": 1, "OF1": 1, "G1": 1,
                "DONE": 1, "QC": 1}
        bars.update(ring_bars(NSLOT))
        n_of = (nkv0, nkv)
        n_roles = 3 + 8 + (1 if copy_q else 0)

        def tile(pre, t, tag):
            return {f"{pre}.{t}.{q}": tag for q in rows}

        def teardown():
            yield ("nbar", "syncthreads", n_roles)

        def producer():
            last = {}
            yield ("load", "Q", 0, dict(tile("Q", 0, "Q"), **tile("Q", 1, "Q")))
            ok = True
            for j in range(nkv):
                for w, nm in enumerate(("K", "V")):
                    idx = 2 * j + w
                    s = idx % NSLOT
                    ok = yield ("twait", f"E{s}", idx // NSLOT - 1, "abort")
                    if not ok:
                        break
                    yield ("load", f"F{s}", idx // NSLOT, {f"kv{s}": f"{nm}({j})"})
                    last[s] = idx // NSLOT
                if not ok:
                    break
            yield ("twait", "Q", 0, "drain")
            for s, ph in last.items():
                yield ("twait", f"F{s}", ph, "drain")
            yield from teardown()

        def gate():
            ok = yield ("twait", "F0", 0, "abort")  # K_0 too (every entry in order)
            if ok:
                yield ("arrive", "G1", 1, 0)
            for j in range(nkv):
                if not ok:
                    break
                v, kn = 2 * j + 1, 2 * j + 2
                ok = yield ("twait", f"F{v % NSLOT}", v // NSLOT, "abort")
                if ok and j + 1 < nkv:
                    ok = yield ("twait", f"F{kn % NSLOT}", kn // NSLOT, "abort")
                for t in (0, 1):
                    if not ok:
                        break
                    if j >= n_of[t]:
                        continue
                    if j > 0:
                        ok = yield ("twait", f"PF{t}", j - 1, "abort")
                    if ok and (t, j) != drop:
                        yield ("arrive", f"PF{t}", 1, j)
                if not ok:
                    break
            yield from teardown()

        def copy():
            ok = yield ("twait", "Q", 0, "abort")
            if ok:
                yield ("read", dict(tile("Q", 0, "Q"), **tile("Q", 1, "Q")))
            yield ("arrive", "QC", 1, 0)  # also after a failed wait
            yield from teardown()

        def qk(t, j):
            slot = (2 * j) % NSLOT
            return ("mma", f"QK({t},{j})", dict(tile("Q", t, "Q"), **{f"kv{slot}": f"K({j})"}),
                    tile("S", t, f"S({t},{j})"))

        def pv(t, j):
            slot = (2 * j + 1) % NSLOT
            reads = dict(tile("S", t, f"P({t},{j})"), **{f"kv{slot}": f"V({j})"})
            if j > 0:
                reads.update(tile("O", t, f"O({t},{j - 1})"))
            return ("mma", f"PV({t},{j})", reads, tile("O", t, f"O({t},{j})"))

        def mma():
            ok = yield ("twait", "Q", 0, "abort")
            if ok:
                ok = yield ("twait", "G1", 0, "abort")
                if ok:
                    yield qk(0, 0)
                    yield ("commit", "SF0", 0)
                    yield qk(1, 0)
                    yield ("commit", "SF1", 0)
                    yield ("commit", "E0", 0)
            for j in range(nkv):
                if not ok:
                    break
                vslot, kidx = (2 * j + 1) % NSLOT, 2 * (j + 1)
                kslot = kidx % NSLOT
                if j < nkv0:
                    ok = yield ("twait", "PF0", j, "abort")
                    if not ok:
                        break
                    yield pv(0, j)
                    if j == nkv0 - 1:
                        yield ("commit", "OF0", 0)
                if j + 1 < nkv0:
                    yield qk(0, j + 1)
                    yield ("commit", "SF0", j + 1)
                ok = yield ("twait", "PF1", j, "abort")
                if not ok:
                    break
                yield pv(1, j)
                yield ("commit", f"E{vslot}", (2 * j + 1) // NSLOT)
                if j == nkv - 1:
                    yield ("commit", "OF1", 0)
                if j + 1 < nkv:
                    yield qk(1, j + 1)
                    yield ("commit", "SF1", j + 1)
                    yield ("commit", f"E{kslot}", kidx // NSLOT)
            yield ("commit", "DONE", 0)
            yield ("twait", "DONE", 0, "drain")
            yield from teardown()

        def softmax(t, q):
            ok = True
            for j in range(n_of[t]):
                ok = yield ("twait", f"SF{t}", j, "abort")
                if not ok:
                    break
                yield ("read", {f"S.{t}.{q}": f"S({t},{j})"})
                yield ("write", {f"S.{t}.{q}": f"P({t},{j})"})
                if j > 0 and rnd.random() < 0.5:  # the lazy rescale of O
                    yield ("read", {f"O.{t}.{q}": f"O({t},{j - 1})"})
                    yield ("write", {f"O.{t}.{q}": f"O({t},{j - 1})"})
                yield ("arrive", f"PF{t}", 32, j)
            ok_e = ok and (yield ("twait", f"OF{t}", 0, "abort"))
            if copy_q:
                ok_e = ok_e and (yield ("twait", "QC", 0, "abort"))
            if ok_e:
                yield ("read", {f"O.{t}.{q}": f"O({t},{n_of[t] - 1})"})
                yield ("write", {f"Q.{t}.{q}": "O out"})  # staging in the Q buffer
            yield ("nbar", f"epilogue{t}", 4)
            yield from teardown()

        roles = {"prod": producer(), "gate": gate(), "mma": mma()}
        if copy_q:
            roles["copy"] = copy()
        for t in (0, 1):
            for q in rows:
                roles[f"s{t}{q}"] = softmax(t, q)
        return bars, roles

    return model


PERSISTENT_TIMEOUT_CASES = [  # (items, ring slots, split_p, sparse, copy_q, stage_q, epi_tma)
    (PERSISTENT_DENSE[0], 4, False, False, True, False, False),
    (PERSISTENT_DENSE[0], 8, True, False, True, False, True),
    (PERSISTENT_DENSE[1], 8, True, False, False, False, True),
    (PERSISTENT_DENSE[2], 4, False, False, False, False, False),
    (PERSISTENT_SPARSE[0], 5, False, True, False, False, False),
    (PERSISTENT_SPARSE[1], 8, True, True, False, False, False),
    ([([0, 2, 3], [1, 2])], 5, False, True, False, True, False),
    ([([], [0, 3])], 8, True, True, False, True, False),
]


@pytest.mark.parametrize("case", range(len(PERSISTENT_TIMEOUT_CASES)))
def test_persistent_forward_without_faults_never_times_out(case):
    items, nslot, split_p, sparse, copy_q, stage_q, epi_tma = PERSISTENT_TIMEOUT_CASES[case]
    for seed in range(20):
        assert not simulate_with_timeouts(
            fwd_persistent_model(items, nslot, split_p, sparse, copy_q, timeouts=True,
                                 stage_q=stage_q, epi_tma=epi_tma), seed, limit=10 ** 6)


@pytest.mark.parametrize("case", range(len(PERSISTENT_TIMEOUT_CASES)))
def test_persistent_forward_any_wait_running_out_ends_the_block_cleanly(case):
    # waits run out at random; whichever do, every role reaches the teardown
    # and nothing is left in flight
    items, nslot, split_p, sparse, copy_q, stage_q, epi_tma = PERSISTENT_TIMEOUT_CASES[case]
    n_failed = 0
    for seed in range(80):
        n_failed += simulate_with_timeouts(
            fwd_persistent_model(items, nslot, split_p, sparse, copy_q, timeouts=True,
                                 stage_q=stage_q, epi_tma=epi_tma), seed, p_spurious=0.01,
            limit=300)
    assert n_failed > 40  # the fault path ran in most schedules


@pytest.mark.parametrize("split_p,drop", [(False, (0, 0)), (False, (1, 3)), (True, (0, 1)),
                                          (True, (1, 4))])
def test_persistent_forward_lost_arrival_is_reported_and_ends_the_block(split_p, drop):
    for seed in range(30):
        assert simulate_with_timeouts(
            fwd_persistent_model(PERSISTENT_DENSE[0], 8 if split_p else 4, split_p, False, True,
                                 timeouts=True, drop=drop), seed, limit=2000)


def test_persistent_forward_exit_without_drain_is_caught():
    caught = False
    for seed in range(40):
        try:
            # copies that take long to land, so some are still in flight when
            # a failed block reaches its teardown
            simulate_with_timeouts(fwd_persistent_model(PERSISTENT_DENSE[0], 4, copy_q=True,
                                                        timeouts=True, mistake="no_drain"),
                                   seed, p_spurious=0.02, limit=300, p_load=0.002)
        except ProtocolError:
            caught = True
            break
    assert caught


FWD_TIMEOUT_SHAPES = [(1, 2, 4), (2, 3, 4), (5, 6, 4), (4, 4, 8)]


@pytest.mark.parametrize("nkv0,nkv,nslot", FWD_TIMEOUT_SHAPES)
def test_forward_without_faults_never_times_out(nkv0, nkv, nslot):
    for seed in range(30):
        failed = simulate_with_timeouts(fwd_timeout_model(nkv0, nkv, nslot), seed, limit=10 ** 6)
        assert not failed


@pytest.mark.parametrize("nkv0,nkv,nslot", FWD_TIMEOUT_SHAPES)
@pytest.mark.parametrize("copy_q", [True, False])
def test_forward_any_wait_running_out_ends_the_block_cleanly(nkv0, nkv, nslot, copy_q):
    # waits run out at random; whichever do, every role reaches the teardown,
    # the epilogue's bar.sync completes and nothing is left in flight
    n_failed = 0
    for seed in range(120):
        n_failed += simulate_with_timeouts(fwd_timeout_model(nkv0, nkv, nslot, copy_q), seed,
                                           p_spurious=0.01, limit=300)
    assert n_failed > 60  # the fault path ran in most schedules


@pytest.mark.parametrize("drop", [(0, 0), (1, 0), (1, 2), (0, 1)])
def test_forward_lost_arrival_is_reported_and_ends_the_block(drop):
    # an arrival on p_full that never comes: the waits on it run out, the
    # failure is recorded, and the block still exits cleanly
    for seed in range(40):
        assert simulate_with_timeouts(fwd_timeout_model(2, 3, 4, drop=drop), seed, limit=2000)


def test_timeout_model_catches_a_partner_left_in_bar_sync():
    # planted: a softmax warp that leaves on a failed wait without reaching
    # the epilogue's bar.sync strands its three partners there
    def model(rnd):
        bars, roles = fwd_timeout_model(2, 3, 4, drop=(1, 1))(rnd)
        inner = roles["s13"]

        def deserter():
            value = None
            while True:
                op = inner.send(value)
                if op[0] == "nbar" and op[1].startswith("epilogue"):
                    return
                value = yield op
        roles["s13"] = deserter()
        return bars, roles

    caught = False
    for seed in range(20):
        try:
            simulate_with_timeouts(model, seed, limit=2000)
        except ProtocolError:
            caught = True
            break
    assert caught
