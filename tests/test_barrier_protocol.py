"""A CPU model of the mbarrier protocol inside attn_kernel (csrc/attention.cu),
run over random unit mixes and random interleavings.  No GPU: each warp role
is a Python generator of the barrier operations it performs, in its order.

Roles and barriers (as in the kernel):
- index warp: claims units into the 3-slot unit ring (U_FULL / U_EMPTY),
  loads each unit's Q (Q_FULL) once the previous unit's products released it
  (Q_EMPTY), and hands each K/V tile's row indices to the copy warps through
  the index ring (I_FULL / I_EMPTY);
- copy warps: fill the K and V stage rings (K_FULL / V_FULL) once the tensor
  core has released the stage (K_EMPTY / V_EMPTY);
- MMA thread: S(j) into buffer b (S_FULL(b)), PV after the buffer's P
  (P_FULL(b)), commits that arrive when its earlier products complete (the
  model completes them after random delays), O_DONE(b) after a unit's last PV;
- softmax warpgroups 0 / 1: wait S_FULL(wg), store P (P_FULL(wg)), wait
  O_DONE(wg) for the epilogue.
Unit kinds: two query tiles ("dual"), one query tile ("one"), and one query
tile split with two key streams, tile j into buffer j & 1 ("two").

Checks: every role finishes (no deadlock); every parity wait passes with its
barrier exactly one phase past what the waiter has consumed, so a parity wait
never aliases a phase two ahead; and every product reads a K or V stage whose
fill for that use has completed.  Planted mistakes must be caught.  The same
model runs the MLA pair kernel's protocol (csrc/mla_pair_kernel.cuh) at the end.
"""
import random

import pytest

NK, NV, NI, RING = 3, 2, 3, 3
NRAW = 4  # raw-code slots of decode over an fp8 pool


class _Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arrivals, self.phase = name, count, 0, 0

    def arrive(self):
        self.arrivals += 1
        assert self.arrivals <= self.count, self.name
        if self.arrivals == self.count:
            self.arrivals = 0
            self.phase += 1


class _Model:
    def __init__(self, units, seed, mistake=None, fp8=False, f16_decode=False,
                 stages=(NK, NV, NI)):
        self.NK, self.NV, self.NI = stages  # K, V and row-index ring depths
        self.rng = random.Random(seed)
        self.units = units
        self.mistake = mistake
        self.fp8 = fp8 or f16_decode  # an fp8 pool: codes converted in shared memory
        # decode over an fp8 pool: the copy warps put the codes into a ring of
        # raw slots (and convert Q); two converting warps fill the stages
        self.f16 = f16_decode
        self.raw = [None] * NRAW  # ("issued" | "landed" | "converted", slot use)
        self.landing = []  # raw slots whose copies are in flight, in issue order
        self.ring = [None] * RING
        self.pending = []  # barriers of the MMA thread's commits, in issue order
        self.bars = {}
        # the query rows of decode over fp8 are converted by both converting groups
        for name, count in [("Q_FULL", 1), ("Q_EMPTY", 1), ("Q_CONV", 2 if f16_decode else 1)]:
            self.bars[name] = _Bar(name, count)
        for b in range(2):
            for name in ("S", "P", "O"):
                self.bars[f"{name}{b}"] = _Bar(f"{name}{b}", 1)
        for s in range(RING):
            self.bars[f"UF{s}"] = _Bar(f"UF{s}", 1)
            # two warpgroups, MMA, copy (+ the two converting groups)
            self.bars[f"UE{s}"] = _Bar(f"UE{s}", 6 if self.f16 else 4)
        for pre, n in (("K", self.NK), ("V", self.NV), ("I", self.NI), ("R", NRAW)):
            for s in range(n):
                self.bars[f"{pre}F{s}"] = _Bar(f"{pre}F{s}", 1)
                self.bars[f"{pre}E{s}"] = _Bar(f"{pre}E{s}", 1)

    def _roles(self):
        roles = {"index": self._index(), "copy": self._copy(), "wg0": self._softmax(0),
                 "wg1": self._softmax(1), "mma": self._mma()}
        if self.f16:
            roles["convert_k"] = self._convert("K")
            roles["convert_v"] = self._convert("V")
        return roles

    def run(self, max_steps=500000):
        roles = self._roles()
        cur = {k: next(g) for k, g in roles.items()}
        done = set()
        for _ in range(max_steps):
            if self.pending and self.rng.random() < 0.3:
                self.bars[self.pending.pop(0)].arrive()  # the oldest product completes
            if self.landing and self.rng.random() < 0.3:  # the oldest raw slot's codes land
                s, use = self.landing.pop(0)
                assert self.raw[s] == ("issued", use)
                self.raw[s] = ("landed", use)
                self.bars[f"RF{s}"].arrive()
            ready = [k for k, op in cur.items() if k not in done and
                     (op[0] != "wait" or (self.bars[op[1]].phase & 1) != op[2])]
            if not ready:
                if self.pending or self.landing:
                    continue
                live = [k for k in cur if k not in done]
                if not live:
                    return
                raise AssertionError("deadlock: " + ", ".join(f"{k} {cur[k]}" for k in live))
            k = self.rng.choice(ready)
            op = cur[k]
            if op[0] == "wait":
                assert self.bars[op[1]].phase == op[3] + 1, f"{k}: {op[1]} aliased"
            elif op[0] == "use":
                assert self.bars[op[1]].phase == op[2] + 1, f"{k}: read {op[1]} before its fill"
            elif op[0] == "arrive":
                self.bars[op[1]].arrive()
            elif op[0] == "commit":
                self.pending.append(op[1])
            elif op[0] == "raw_issue":  # the copies of slot use op[2] into slot op[1]
                assert self.raw[op[1]] in (None, ("converted", op[2] - NRAW)), \
                    f"{k}: raw slot {op[1]} overwritten before its conversion"
                self.raw[op[1]] = ("issued", op[2])
                self.landing.append((op[1], op[2]))
            elif op[0] == "raw_convert":
                assert self.raw[op[1]] == ("landed", op[2]), f"{k}: raw slot converted before it landed"
                self.raw[op[1]] = ("converted", op[2])
            try:
                cur[k] = next(roles[k])
            except StopIteration:
                done.add(k)
        raise AssertionError("step limit")

    @staticmethod
    def _wait(bar, consumed):
        return ("wait", bar, consumed & 1, consumed)

    def _units(self):
        full = [0] * RING
        uc = 0
        while True:
            s = uc % RING
            yield self._wait(f"UF{s}", full[s])
            full[s] += 1
            u = self.ring[s]
            yield ("arrive", f"UE{s}")
            yield ("unit", u)
            if u is None:
                return
            uc += 1

    def _index(self):
        q_cnt = ic = 0
        for uc, u in enumerate(self.units + [None]):
            s = uc % RING
            if uc >= RING:
                yield self._wait(f"UE{s}", uc // RING - 1)
            self.ring[s] = u
            yield ("arrive", f"UF{s}")
            if u is None:
                return
            if u["nt"] == 0:
                continue
            if q_cnt > 0:
                yield self._wait("Q_EMPTY", q_cnt - 1)
            yield ("arrive", "Q_FULL")
            q_cnt += 1
            for _ in range(u["nt"]):
                si = ic % self.NI
                if ic >= self.NI:
                    yield self._wait(f"IE{si}", ic // self.NI - 1)
                yield ("arrive", f"IF{si}")
                ic += 1

    def _copy(self):
        if self.f16:
            yield from self._copy_raw()
            return
        if self.fp8:
            yield from self._copy_fp8()
            return
        kc = vc = ic = 0
        for op in self._units():
            if op[0] != "unit":
                yield op
                continue
            if op[1] is None:
                return
            for _ in range(op[1]["nt"]):
                si = ic % self.NI
                yield self._wait(f"IF{si}", ic // self.NI)
                yield ("arrive", f"IE{si}")
                ic += 1
                ks, vs = kc % self.NK, vc % self.NV
                if kc >= self.NK:
                    yield self._wait(f"KE{ks}", kc // self.NK - 1)
                yield ("arrive", f"KF{ks}")
                kc += 1
                if vc >= self.NV and self.mistake != "V refilled before release":
                    yield self._wait(f"VE{vs}", vc // self.NV - 1)
                yield ("arrive", f"VF{vs}")
                vc += 1

    def _copy_raw(self):
        """Decode over an fp8 pool: per tile, the codes of K(j) and of V(j)
        go into the next two raw slots once the converting warps have read
        what those slots held."""
        rc = ic = 0
        for op in self._units():
            if op[0] != "unit":
                yield op
                continue
            u = op[1]
            if u is None:
                return
            for j in range(u["nt"]):
                si = ic % self.NI
                yield self._wait(f"IF{si}", ic // self.NI)
                yield ("arrive", f"IE{si}")
                ic += 1
                for _ in range(2):  # K(j), V(j)
                    s = rc % NRAW
                    if rc >= NRAW and self.mistake != "raw slot reused before its conversion":
                        yield self._wait(f"RE{s}", rc // NRAW - 1)
                    yield ("raw_issue", s, rc)
                    rc += 1

    def _convert(self, pre):
        """A converting group (K or V slots): the unit's query rows (Q_CONV,
        with the other group), then its raw slots in order (K(j) in use 2j,
        V(j) in use 2j + 1), each into the next stage of its ring once the
        codes have landed and the tensor core has released the stage."""
        rc = 0 if pre == "K" else 1
        cnt = qc = 0
        n = self.NK if pre == "K" else self.NV
        for op in self._units():
            if op[0] != "unit":
                yield op
                continue
            u = op[1]
            if u is None:
                return
            if u["nt"] == 0:
                continue
            yield self._wait("Q_FULL", qc)
            qc += 1
            yield ("arrive", "Q_CONV")
            for _ in range(u["nt"]):
                s = rc % NRAW
                if self.mistake != "raw slot converted before it landed":
                    yield self._wait(f"RF{s}", rc // NRAW)
                if cnt >= n:
                    yield self._wait(f"{pre}E{cnt % n}", cnt // n - 1)
                yield ("raw_convert", s, rc)
                yield ("arrive", f"{pre}F{cnt % n}")
                yield ("arrive", f"RE{s}")
                rc += 2
                cnt += 1

    def _copy_fp8(self):
        """The fp8-pool order: a tile's codes are issued, and converted (then
        the stage's full barrier) only after the next tile's codes are issued:
        K(0), V(0), the query rows' conversion, then per tile K(j+1),
        convert K(j), V(j+1), convert V(j)."""
        kc = vc = ic = qc = 0

        def fetch():
            nonlocal ic
            si = ic % self.NI
            yield self._wait(f"IF{si}", ic // self.NI)
            yield ("arrive", f"IE{si}")
            ic += 1

        def issue(pre, cnt, n):  # wait until the stage is free again
            if cnt >= n:
                yield self._wait(f"{pre}E{cnt % n}", cnt // n - 1)

        for op in self._units():
            if op[0] != "unit":
                yield op
                continue
            u = op[1]
            if u is None:
                return
            nt = u["nt"]
            if nt == 0:
                continue
            if (self.NK < 2 or self.NV < 2) and self.mistake != "one stage converted one tile behind":
                # one K or one V stage (the 288 / 256 layout): a tile's codes
                # are converted as soon as they land, before the next tile
                for _ in range(nt):
                    yield from fetch()
                    yield from issue("K", kc, self.NK)
                    yield ("arrive", f"KF{kc % self.NK}")
                    kc += 1
                    yield from issue("V", vc, self.NV)
                    yield ("arrive", f"VF{vc % self.NV}")
                    vc += 1
                continue
            yield from fetch()
            yield from issue("K", kc, self.NK)
            yield from issue("V", vc, self.NV)
            if self.f16:
                yield self._wait("Q_FULL", qc)
                qc += 1
                yield ("arrive", "Q_CONV")
            for j in range(nt):
                more = j + 1 < nt
                if more:
                    yield from fetch()
                    yield from issue("K", kc + 1, self.NK)
                yield ("arrive", f"KF{kc % self.NK}")
                kc += 1
                if more:
                    yield from issue("V", vc + 1, self.NV)
                yield ("arrive", f"VF{vc % self.NV}")
                vc += 1

    def _softmax(self, wg):
        s_cnt = o_cnt = 0
        for op in self._units():
            if op[0] != "unit":
                yield op
                continue
            u = op[1]
            if u is None:
                return
            two = u["kind"] == "two"
            if not two and wg == 1 and u["kind"] == "one":
                continue  # one query tile: warpgroup 1 has no rows
            j0, step = (wg, 2) if two else (0, 1)
            if u["nt"] - j0 <= 0:
                continue  # no tile of this stream: zero partial, no barrier
            for _ in range(j0, u["nt"], step):
                yield self._wait(f"S{wg}", s_cnt)
                s_cnt += 1
                yield ("arrive", f"P{wg}")
            yield self._wait(f"O{wg}", o_cnt)
            o_cnt += 1

    def _mma(self):
        q_cnt = kc = vc = 0
        p = [0, 0]
        shared_p = self.mistake == "shared P counter"

        def wait_p(b):
            i = 0 if shared_p else b
            op = self._wait(f"P{b}", p[i])
            p[i] += 1
            return op

        for op in self._units():
            if op[0] != "unit":
                yield op
                continue
            u = op[1]
            if u is None:
                return
            nt = u["nt"]
            if nt == 0:
                continue
            yield self._wait("Q_CONV" if self.f16 else "Q_FULL", q_cnt)
            q_cnt += 1
            if u["kind"] == "two":
                # S(j) into buffer j & 1 waits only for PV(j - 2)
                for j in range(nt):
                    b = j & 1
                    if j >= 2:
                        vs = vc % self.NV
                        yield self._wait(f"VF{vs}", vc // self.NV)
                        yield wait_p(b)
                        yield ("use", f"VF{vs}", vc // self.NV)
                        yield ("commit", f"VE{vs}")
                        vc += 1
                    ks = kc % self.NK
                    yield self._wait(f"KF{ks}", kc // self.NK)
                    yield ("use", f"KF{ks}", kc // self.NK)
                    yield ("commit", f"S{b}")
                    yield ("commit", f"KE{ks}")
                    kc += 1
                    if j == nt - 1 and self.mistake != "no Q release":
                        yield ("commit", "Q_EMPTY")
                for j in range(max(nt - 2, 0), nt):
                    vs = vc % self.NV
                    yield self._wait(f"VF{vs}", vc // self.NV)
                    yield wait_p(j & 1)
                    yield ("use", f"VF{vs}", vc // self.NV)
                    yield ("commit", f"O{j & 1}")
                    yield ("commit", f"VE{vs}")
                    vc += 1
                continue
            q1 = u["kind"] == "dual"
            ks = kc % self.NK
            yield self._wait(f"KF{ks}", kc // self.NK)
            yield ("commit", "S0")
            if q1:
                yield ("commit", "S1")
            yield ("commit", f"KE{ks}")
            kc += 1
            if nt == 1:
                yield ("commit", "Q_EMPTY")
            for j in range(1, nt):
                ks, vs = kc % self.NK, vc % self.NV
                yield self._wait(f"KF{ks}", kc // self.NK)
                yield self._wait(f"VF{vs}", vc // self.NV)
                yield wait_p(0)
                yield ("use", f"KF{ks}", kc // self.NK)
                yield ("use", f"VF{vs}", vc // self.NV)
                yield ("commit", "S0")
                if q1:
                    yield wait_p(1)
                    yield ("commit", "S1")
                yield ("commit", f"VE{vs}")
                vc += 1
                yield ("commit", f"KE{ks}")
                kc += 1
                if j == nt - 1:
                    yield ("commit", "Q_EMPTY")
            vs = vc % self.NV
            yield self._wait(f"VF{vs}", vc // self.NV)
            yield wait_p(0)
            yield ("use", f"VF{vs}", vc // self.NV)
            yield ("commit", "O0")
            if q1:
                yield wait_p(1)
                yield ("commit", "O1")
            yield ("commit", f"VE{vs}")
            vc += 1


def _random_units(rng, n):
    return [{"kind": rng.choice(["dual", "one", "two"]),
             "nt": rng.choice([0, 1, 1, 2, 3, 4, 5, 7])} for _ in range(n)]


def _trials(n, mistake=None):
    rng = random.Random(1)
    for t in range(n):
        _Model(_random_units(rng, rng.randint(1, 12)), seed=t, mistake=mistake).run()


def test_fp8_protocols_have_no_deadlock_and_no_parity_aliasing():
    """An fp8 pool: extend units of every kind with the fp8 copy order, and
    decode units (two key streams, or one stream when the workspace holds one
    partial slot per unit) whose query rows the copy warps convert to f16."""
    rng = random.Random(3)
    for t in range(150):
        _Model(_random_units(rng, rng.randint(1, 12)), seed=t, fp8=True).run()
    for t in range(300):
        # K stage 0 holds raw slots: 2 K stages for 128 dims, 4 for 64
        stages = (2, 2, 3) if t % 2 else (4, 5, 4)
        kind = rng.choice(["two", "one"])
        units = [{"kind": kind, "nt": rng.choice([0, 1, 2, 3, 6])} for _ in range(rng.randint(1, 10))]
        _Model(units, seed=t, f16_decode=True, stages=stages).run()


def test_split_head_dim_fp8_protocol():
    """The split head dims over an fp8 pool (extend): 192 / 128 (two stages
    each) converts a tile after the next one is issued; 288 / 256 (one stage
    each) converts a tile as soon as it lands, since the one-behind order
    would wait for its own stage."""
    rng = random.Random(8)
    for stages in ((2, 2, 3), (1, 1, 3)):
        for t in range(150):
            units = [{"kind": "one", "nt": rng.choice([0, 1, 2, 3, 5, 8])}
                     for _ in range(rng.randint(1, 12))]
            _Model(units, seed=t, fp8=True, stages=stages).run()
    with pytest.raises(AssertionError):  # the one-behind order on one stage deadlocks
        for t in range(150):
            units = [{"kind": "one", "nt": rng.choice([1, 2, 3])} for _ in range(rng.randint(1, 6))]
            _Model(units, seed=t, fp8=True, stages=(1, 1, 3),
                   mistake="one stage converted one tile behind").run()


@pytest.mark.parametrize("mistake", ["raw slot reused before its conversion",
                                     "raw slot converted before it landed"])
def test_fp8_decode_model_catches_planted_mistakes(mistake):
    rng = random.Random(4)
    with pytest.raises(AssertionError):
        for t in range(150):
            units = [{"kind": "two", "nt": rng.choice([1, 2, 3, 6])} for _ in range(rng.randint(1, 10))]
            _Model(units, seed=t, f16_decode=True, stages=(2, 2, 3), mistake=mistake).run()


def test_protocol_has_no_deadlock_and_no_parity_aliasing():
    _trials(150)


@pytest.mark.parametrize("stages", [(2, 2, 3), (1, 1, 3)])
def test_split_head_dim_protocol(stages):
    """The split head dims (Lq / Lv = 192 / 128 with two K and two V stages,
    288 / 256 with one of each): every unit has one query tile and one key
    stream (warpgroup 1 idles), so only "one" units occur."""
    rng = random.Random(7)
    for t in range(200):
        units = [{"kind": "one", "nt": rng.choice([0, 1, 2, 3, 5, 8])}
                 for _ in range(rng.randint(1, 12))]
        _Model(units, seed=t, stages=stages).run()


@pytest.mark.parametrize("mistake", ["shared P counter", "no Q release",
                                     "V refilled before release"])
def test_model_catches_planted_mistakes(mistake):
    with pytest.raises(AssertionError):
        _trials(150, mistake)


# ------------------------------------------------------------------ MLA kernel
class _MlaPairModel:
    """The mbarrier protocol of mla_pair_kernel (csrc/mla_pair_kernel.cuh):
    two CTAs of a cluster take the same units in the same order.  A claiming
    thread of CTA 0 writes each unit into slot uc % 4 of both CTAs' unit
    rings (U_FULL of each CTA); every role releases the slot on its own CTA's
    U_EMPTY, and a forwarding thread of CTA 1 passes each completed phase of
    CTA 1's U_EMPTY on to CTA 0's (one more arrival there).  The claimer
    publishes unit uc once every role of both CTAs has taken unit uc - 2, so
    a unit is never overwritten before all eight roles have read it.  The softmax writes a unit's Q after the previous unit's
    epilogue (or, in decode of at most 32 rows, the MMA warp writes it as it
    starts the unit: it has waited for the previous unit's last P, which the
    softmax writes only after the last QK^T landed); the model tracks which
    unit's Q each CTA holds and the QK^T products in flight that read it.
    Per CTA: one K ring of four stages (the tile is also V); QK^T runs
    two tiles ahead of PV, S is read and released early (S_FREE); P and O are
    reused after each PV (PV_DONE), whose phases the softmax counts across
    units (pv_base).

    The partial S of each tile goes to the other CTA one tile ahead of its
    softmax, into receive buffer t & 1: the softmax reads S(t), releases it
    and stores its partial there asynchronously; the bytes land later and
    complete the other CTA's XFULL of the buffer, which its thread 0 arms
    (one arrival) once the buffer's previous phase has completed.  The
    softmax of tile t then adds the received partial to its own.  No barrier
    frees a buffer; the model checks every buffer write and read against the
    buffer's state, so a send that could overwrite an unread tile fails."""
    NK, NI, R, AHEAD = 4, 4, 4, 2
    ROLES = {"index", "copy", "softmax", "mma"}

    def __init__(self, units, seed, mistake=None, fp8=False, lead=1, mma_q=False, raw=False):
        self.mma_q = mma_q  # the MMA warp writes Q (decode of at most 32 rows)
        # decode over an fp8 pool, at most 32 rows: each copy thread stages
        # its codes in a ring of NRAW private raw slots and converts a tile
        # into one of three stages NRAW - 1 tiles later, across units
        self.raw = raw
        if raw:
            self.NK, self.NRAW = 3, 4
            self.rawslot = {(c, r): None for c in (0, 1) for r in range(self.NRAW)}
        self.rng = random.Random(seed)
        self.units, self.mistake = units, mistake
        self.lead = lead  # CTA 0's roles are picked this many times as often
        # unit ring slot (CTA, slot) -> (claim number, unit, roles that read it)
        self.uring = {(c, s): None for c in (0, 1) for s in range(self.R)}
        self.q_unit = {0: None, 1: None}   # whose Q the CTA's TMEM holds
        self.q_readers = {0: 0, 1: 0}      # QK^T products in flight
        # an fp8 pool: the copy warps mark tile j full only after issuing
        # tile j + 1 (they convert tile j's codes in place in between)
        self.fp8 = fp8
        self.pending = {0: [], 1: []}
        self.xbuf = {(c, b): None for c in (0, 1) for b in (0, 1)}  # ("written" | "read", tile)
        self.bars = {}
        for c in (0, 1):
            for n in ("Q_FULL", "S_FULL", "P_FULL", "O_DONE", "S_FREE", "PV_DONE"):
                self.bars[f"{c}{n}"] = _Bar(f"{c}{n}", 1)
            for b in (0, 1):  # the local arm + the stores' bytes
                self.bars[f"{c}XFULL{b}"] = _Bar(f"{c}XFULL{b}", 2)
            for pre, n in (("K", self.NK), ("I", self.NI)):
                for s in range(n):
                    self.bars[f"{c}{pre}F{s}"] = _Bar(f"{c}{pre}F{s}", 1)
                    self.bars[f"{c}{pre}E{s}"] = _Bar(f"{c}{pre}E{s}", 1)
            for s in range(self.R):
                self.bars[f"{c}UF{s}"] = _Bar(f"{c}UF{s}", 1)
                # CTA 0: its four roles and the forwarder; CTA 1: its four roles
                self.bars[f"{c}UE{s}"] = _Bar(f"{c}UE{s}", 5 if c == 0 else 4)

    @staticmethod
    def _wait(bar, consumed):
        return ("wait", bar, consumed & 1, consumed)

    def run(self, max_steps=500000):
        def ending(gen):  # every role ends with a no-op (a role may have no work)
            yield from gen
            yield ("end",)

        roles = {"0claim": ending(self._claim()), "1forward": ending(self._forward())}
        for c in (0, 1):
            roles[f"{c}index"] = ending(self._index(c))
            roles[f"{c}copy"] = ending(self._copy(c))
            roles[f"{c}softmax"] = ending(self._softmax(c))
            roles[f"{c}mma"] = ending(self._mma(c))
        cur = {k: next(g) for k, g in roles.items()}
        done = set()
        for _ in range(max_steps):
            for c in (0, 1):
                if self.pending[c] and self.rng.random() < 0.3:
                    ev = self.pending[c].pop(0)
                    if isinstance(ev, tuple):  # stored bytes land in CTA ev[1], buffer ev[2] & 1
                        key = (ev[1], ev[2] & 1 if self.mistake != "one receive buffer" else 0)
                        state = self.xbuf[key]
                        assert state is None or state[0] == "read", "buffer overwritten"
                        self.xbuf[key] = ("written", ev[2])
                        self.bars[f"{ev[1]}XFULL{ev[2] & 1}"].arrive()
                    else:
                        if ev.endswith("S_FULL"):  # the QK^T landed: its Q reads are done
                            self.q_readers[int(ev[0])] -= 1
                        self.bars[ev].arrive()
            ready = [k for k, op in cur.items() if k not in done and
                     (op[0] != "wait" or (self.bars[op[1]].phase & 1) != op[2])]
            if not ready:
                if self.pending[0] or self.pending[1]:
                    continue
                live = [k for k in cur if k not in done]
                if not live:
                    return
                raise AssertionError("deadlock: " + ", ".join(f"{k} {cur[k]}" for k in live))
            k = self.rng.choices(ready, [self.lead if r[0] == "0" else 1 for r in ready])[0]
            op = cur[k]
            if op[0] == "wait":
                assert self.bars[op[1]].phase == op[3] + 1, f"{k}: {op[1]} aliased"
            elif op[0] == "use":
                assert self.bars[op[1]].phase == op[2] + 1, f"{k}: read {op[1]} before its fill"
            elif op[0] == "arrive":
                self.bars[op[1]].arrive()
            elif op[0] == "commit":
                self.pending[int(op[1][0])].append(op[1])
            elif op[0] == "send":  # asynchronous stores into the other CTA; they land later
                self.pending[op[1]].append(("land", 1 - op[1], op[2]))
            elif op[0] == "writeq":  # the softmax writes unit op[2]'s Q into CTA op[1]'s TMEM
                assert self.q_readers[op[1]] == 0, f"{k}: Q overwritten under a QK^T in flight"
                self.q_unit[op[1]] = op[2]
            elif op[0] == "qk":  # a QK^T of unit op[2] reads CTA op[1]'s Q
                assert self.q_unit[op[1]] == op[2], f"{k}: QK^T of unit {op[2]} reads another unit's Q"
                self.q_readers[op[1]] += 1
            elif op[0] == "raw_put":  # codes of tile op[2] into raw slot op[2] % NRAW of CTA op[1]
                key = (op[1], op[2] % self.NRAW)
                prev = self.rawslot[key]
                assert prev is None or prev == ("converted", op[2] - self.NRAW), \
                    f"{k}: raw slot overwritten before its conversion"
                self.rawslot[key] = ("issued", op[2])
            elif op[0] == "raw_take":  # tile op[2] converted out of its raw slot
                key = (op[1], op[2] % self.NRAW)
                assert self.rawslot[key] == ("issued", op[2]), f"{k}: raw slot does not hold the tile"
                self.rawslot[key] = ("converted", op[2])
            elif op[0] == "publish":  # the claimer writes unit use op[2] into slot op[1] of both CTAs
                for c in (0, 1):
                    prev = self.uring[(c, op[1])]
                    assert prev is None or prev[2] == self.ROLES, \
                        f"unit slot {op[1]} of CTA {c} overwritten before all its roles read it"
                    self.uring[(c, op[1])] = (op[2], op[3], set())
            elif op[0] == "combine":  # the softmax reads the received partial of tile op[2]
                key = (op[1], op[2] & 1 if self.mistake != "one receive buffer" else 0)
                assert self.xbuf[key] == ("written", op[2]), f"{k}: partial read before it lands"
                self.xbuf[key] = ("read", op[2])
            try:
                cur[k] = next(roles[k])
            except StopIteration:
                done.add(k)
        raise AssertionError("step limit")

    def _claim(self):
        ahead = self.AHEAD
        for uc, u in enumerate(self.units + [None]):
            s = uc % self.R
            if uc >= ahead:  # every role took unit uc - ahead (and so uc - R)
                e = uc - ahead
                yield self._wait(f"0UE{e % self.R}", e // self.R)
            yield ("publish", s, uc, u)
            yield ("arrive", "0UF" + str(s))  # local
            yield ("arrive", "1UF" + str(s))  # remote, after the remote store
            if u is None:
                return

    def _forward(self):
        """CTA 1's forwarder: each completed phase of CTA 1's U_EMPTY becomes
        one arrival on CTA 0's, up to the end marker."""
        for uc in range(len(self.units) + 1):
            s = uc % self.R
            if self.mistake != "forwarder arrives before CTA 1's roles read the slot":
                yield self._wait(f"1UE{s}", uc // self.R)
            yield ("arrive", f"0UE{s}")

    def _take(self, c, role, uc):
        """Unit use uc from this CTA's ring: wait, read, release locally."""
        s = uc % self.R
        yield self._wait(f"{c}UF{s}", uc // self.R)
        val = self.uring[(c, s)]
        assert val is not None and val[0] == uc, f"{c}{role}: unit slot {s} does not hold use {uc}"
        val[2].add(role)
        yield ("arrive", f"{c}UE{s}")

    def _index(self, c):
        ic = 0
        for uc, u in enumerate(self.units):
            yield from self._take(c, "index", uc)
            for _ in range(u["nt"]):
                si = ic % self.NI
                if ic >= self.NI:
                    yield self._wait(f"{c}IE{si}", ic // self.NI - 1)
                yield ("arrive", f"{c}IF{si}")
                ic += 1
        yield from self._take(c, "index", len(self.units))

    def _copy(self, c):
        kc = ic = 0

        def issue():
            nonlocal kc, ic
            si = ic % self.NI
            yield self._wait(f"{c}IF{si}", ic // self.NI)
            yield ("arrive", f"{c}IE{si}")
            ic += 1
            ks = kc % self.NK
            if kc >= self.NK:
                yield self._wait(f"{c}KE{ks}", kc // self.NK - 1)
            kc += 1

        if self.raw:
            issued = conv = 0

            def convert():
                nonlocal conv
                ks = conv % self.NK
                if conv >= self.NK and self.mistake != "stage converted into before its release":
                    yield self._wait(f"{c}KE{ks}", conv // self.NK - 1)
                yield ("raw_take", c, conv)
                yield ("arrive", f"{c}KF{ks}")
                conv += 1

            lag = self.NRAW if self.mistake == "raw slot reused before its conversion" else self.NRAW - 1
            for uc, u in enumerate(self.units):
                yield from self._take(c, "copy", uc)
                for _ in range(u["nt"]):
                    si = ic % self.NI
                    yield self._wait(f"{c}IF{si}", ic // self.NI)
                    yield ("arrive", f"{c}IE{si}")
                    ic += 1
                    yield ("raw_put", c, issued)
                    issued += 1
                    if issued - conv > lag:
                        yield from convert()
                # the unit's last tiles before the next unit: its claim may
                # wait for this unit's products, which wait for these tiles
                if self.mistake != "conversions carried across units":
                    while conv < issued:
                        yield from convert()
            while conv < issued:
                yield from convert()
            yield from self._take(c, "copy", len(self.units))
            return
        for uc, u in enumerate(self.units):
            yield from self._take(c, "copy", uc)
            nt = u["nt"]
            if not self.fp8:
                for _ in range(nt):
                    yield from issue()
                    yield ("arrive", f"{c}KF{(kc - 1) % self.NK}")
                continue
            if nt == 0:
                continue
            yield from issue()
            for j in range(nt):
                st_j = (kc - 1) % self.NK
                if j + 1 < nt:
                    yield from issue()
                yield ("arrive", f"{c}KF{st_j}")
        yield from self._take(c, "copy", len(self.units))

    def _softmax(self, c):
        s_cnt = o_cnt = pv_base = n_sent = n_recv = 0

        def send():
            nonlocal s_cnt, n_sent
            yield self._wait(f"{c}S_FULL", s_cnt)
            s_cnt += 1
            yield ("arrive", f"{c}S_FREE")
            yield ("send", c, n_sent)
            n_sent += 1

        def combine():
            nonlocal n_recv
            b = n_recv & 1
            early = self.mistake == "next phase armed before the wait"
            if early:
                yield ("arrive", f"{c}XFULL{b}")
            if self.mistake != "partial read before it lands":
                yield self._wait(f"{c}XFULL{b}", n_recv >> 1)
            if not early:
                yield ("arrive", f"{c}XFULL{b}")  # arm the buffer's phase for tile n_recv + 2
            yield ("combine", c, n_recv)
            n_recv += 1

        yield ("arrive", f"{c}XFULL0")  # arm the first two tiles' phases
        yield ("arrive", f"{c}XFULL1")
        early = self.mistake == "next Q written before the last QK landed"
        q_in = taken = False  # (planted mistake) the next unit taken and its Q written early
        for uc, u in enumerate(self.units):
            if not taken:
                yield from self._take(c, "softmax", uc)
            taken = False
            nt = u["nt"]
            if nt == 0:
                q_in = False
                continue
            if not q_in and not self.mma_q:
                yield ("writeq", c, uc)
                yield ("arrive", f"{c}Q_FULL")  # this CTA's Q dims written into TMEM
            q_in = False
            yield from send()
            for j in range(nt):
                if early and j == 0:
                    yield from self._take(c, "softmax", uc + 1)
                    taken = True
                    if uc + 1 < len(self.units) and self.units[uc + 1]["nt"] > 0:
                        yield ("writeq", c, uc + 1)
                        yield ("arrive", f"{c}Q_FULL")
                        q_in = True
                yield from combine()
                if j + 1 < nt:
                    yield from send()
                if j > 0 and self.mistake != "P written before the previous PV":
                    yield self._wait(f"{c}PV_DONE", pv_base + j - 1)
                yield ("arrive", f"{c}P_FULL")
            yield self._wait(f"{c}O_DONE", o_cnt)
            o_cnt += 1
            if self.mistake != "PV count not carried across units":
                pv_base += nt
        if not taken:
            yield from self._take(c, "softmax", len(self.units))

    def _mma(self, c):
        q_cnt = kc = s_free = p_cnt = 0
        cur = None
        early_q = False  # (planted mistake) the next unit's Q written after the last QK^T issue
        nxt = {}
        for i, u in enumerate(self.units):  # the next unit with tiles
            nxt[i] = next((k for k in range(i + 1, len(self.units)) if self.units[k]["nt"] > 0), None)

        def qk(kpos):
            nonlocal early_q
            yield self._wait(f"{c}KF{kpos % self.NK}", kpos // self.NK)
            yield ("use", f"{c}KF{kpos % self.NK}", kpos // self.NK)
            yield ("qk", c, cur)
            yield ("commit", f"{c}S_FULL")
            if (self.mma_q and self.mistake == "next Q written after the last QK issue"
                    and kpos == k_last and nxt[cur] is not None):
                yield ("writeq", c, nxt[cur])
                early_q = True

        for uc, u in enumerate(self.units):
            yield from self._take(c, "mma", uc)
            nt = u["nt"]
            if nt == 0:
                continue
            cur = uc
            if self.mma_q:
                if not early_q:
                    yield ("writeq", c, uc)
                early_q = False
            else:
                yield self._wait(f"{c}Q_FULL", q_cnt)
            q_cnt += 1
            k0 = kc
            k_last = k0 + nt - 1
            yield from qk(k0)
            yield self._wait(f"{c}S_FREE", s_free)
            s_free += 1
            if nt > 1:
                yield from qk(k0 + 1)
            for j in range(nt):
                if j + 1 < nt:
                    yield self._wait(f"{c}S_FREE", s_free)
                    s_free += 1
                    if j + 2 < nt:
                        yield from qk(k0 + j + 2)
                yield self._wait(f"{c}P_FULL", p_cnt)
                p_cnt += 1
                yield ("use", f"{c}KF{(k0 + j) % self.NK}", (k0 + j) // self.NK)  # V = the K tile
                yield ("commit", f"{c}PV_DONE")
                yield ("commit", f"{c}KE{(k0 + j) % self.NK}")
            kc = k0 + nt
            yield ("commit", f"{c}O_DONE")
        yield from self._take(c, "mma", len(self.units))


def _mla_trials(n, mistake=None, mma_q=False, raw=False):
    rng = random.Random(2)
    for t in range(n):
        # every third trial has runs of empty units, which the softmax of one
        # CTA passes without an exchange (so it can run ahead of the other)
        sizes = [0, 0, 0, 1, 2, 5] if t % 3 == 2 else [0, 1, 1, 2, 3, 5, 8]
        units = [{"nt": rng.choice(sizes)} for _ in range(rng.randint(1, 12))]
        # and in every other one CTA 0 runs ahead
        _MlaPairModel(units, seed=t, mistake=mistake, lead=8 if t % 2 else 1, mma_q=mma_q,
                      raw=raw).run()


def test_mla_protocol_has_no_deadlock_and_no_parity_aliasing():
    _mla_trials(150)


def test_mla_small_group_decode_protocol():
    """Decode of at most 32 rows: the MMA warp writes each unit's Q itself."""
    _mla_trials(150, mma_q=True)


def test_mla_small_group_fp8_decode_protocol():
    """... and over an fp8 pool: codes staged in private raw slots, converted
    into one of three stages three tiles later; a unit's last tiles are
    converted before the next unit is taken (carried across units, they
    deadlock: the next claim waits for this unit's products)."""
    _mla_trials(150, mma_q=True, raw=True)


@pytest.mark.parametrize("mistake", ["raw slot reused before its conversion",
                                     "stage converted into before its release",
                                     "conversions carried across units"])
def test_mla_raw_ring_model_catches_planted_mistakes(mistake):
    with pytest.raises(AssertionError):
        _mla_trials(150, mistake, mma_q=True, raw=True)


def test_mla_model_catches_q_written_under_products():
    with pytest.raises(AssertionError):
        _mla_trials(150, "next Q written after the last QK issue", mma_q=True)


def test_mla_fp8_protocol_has_no_deadlock_and_no_parity_aliasing():
    """An fp8 pool: tile j's stage becomes full after tile j + 1's copies."""
    rng = random.Random(5)
    for t in range(150):
        units = [{"nt": rng.choice([0, 1, 1, 2, 3, 5, 8])} for _ in range(rng.randint(1, 10))]
        _MlaPairModel(units, seed=t, fp8=True).run()


@pytest.mark.parametrize("mistake", ["P written before the previous PV",
                                     "PV count not carried across units",
                                     "partial read before it lands",
                                     "next phase armed before the wait",
                                     "one receive buffer",
                                     "forwarder arrives before CTA 1's roles read the slot",
                                     "next Q written before the last QK landed"])
def test_mla_model_catches_planted_mistakes(mistake):
    with pytest.raises(AssertionError):
        _mla_trials(150, mistake)
