"""A model of the tensor-core coarse pass's mbarrier protocol (csrc/coarse_tc.cu), run on the CPU.

Every role of one CTA follows the kernel's loops over its rings: the producer (packed stages and
B quarters in one fixed order), the three MMA issuers (each owning every third B quarter), the
eight dequantising warps (four lane quadrants x two chunk parities), the fold warps and the
selection warps. Copies and tcgen05 commits complete asynchronously, at random later points
(a thread's commits in order). A scheduler interleaves everything at random and checks:

* no deadlock: some role or completion can always move until every role is done;
* no phase aliasing: an mbarrier wait is a parity test, so when it is evaluated the barrier must
  be on the awaited phase or the one after it; every arrival must land on the phase it is meant
  for (an arrival one phase early would complete the wrong phase).

The constants are read from the kernel source, so a change there is modelled here. Mutated
protocols (a miscounted ring, a missing release wait) must fail the same checks.
"""
import os
import random
import re

import pytest

SRC = os.path.join(os.path.dirname(__file__), "..", "bit_draft_lm_gb300", "csrc", "coarse_tc.cu")


def _constants():
    text = open(SRC).read()
    out = {}
    for name in ("kWNB", "kWIssuers", "kWMaxNA", "kWTmemCols", "kWDeqWarps", "kWFoldWarps",
                 "kWSelWarps", "kWMaxNP", "kWStageBytes"):
        m = re.search(r"constexpr int %s = (\d+);" % name, text)
        assert m, name
        out[name] = int(m.group(1))
    return out


C = _constants()


class Deadlock(Exception):
    pass


class Aliasing(Exception):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.done, self.pending = name, count, 0, 0

    def arrive(self, phase):
        if phase != self.done:
            raise Aliasing(f"{self.name}: arrival meant for phase {phase} while on {self.done}")
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.done += 1

    def ready(self, phase):
        # the hardware test: parity of the awaited phase against the barrier's current phase
        if not (phase <= self.done <= phase + 1):
            raise Aliasing(f"{self.name}: wait for phase {phase} evaluated on phase {self.done}")
        return self.done == phase + 1


def _geometry(G, NCOL, K, tiles, np_):
    CPJ = G // 16
    CPQ = CPJ // 4
    NAS = min((C["kWTmemCols"] - C["kWIssuers"] * NCOL) // 32, C["kWMaxNA"]) & ~1
    assert NAS % CPQ == 0 and NAS // CPQ >= 2
    RB = K // 4
    return dict(CPJ=CPJ, CPQ=CPQ, NAS=NAS, NAQ=NAS // CPQ, NJ=RB // G,
                NS=RB // C["kWStageBytes"], T=tiles, np=np_)


# each role is a generator of actions: ("wait", bar, phase), ("arrive", bar, phase),
# ("copy", bar, phase) (completes later) and ("commit", queue, bar, phase) (completes later, in
# order per queue)

def producer(g, mutant):
    np_, NS, T = g["np"], g["NS"], g["T"]
    total = T * NS
    kqps = 8 // g["CPQ"]
    qpt = g["NJ"] * 4 * (4 if mutant == "quarters_per_tile_x_planes" else 1)
    nb = C["kWNB"]
    issued = issued_b = 0
    bunit = 0
    for gs in range(1 - np_, total):
        if issued < total:
            if issued >= np_:
                yield ("wait", f"pempty{issued % np_}", issued // np_ - 1)
            yield ("arrive", f"pfull{issued % np_}", issued // np_)
            yield ("copy", f"pfull{issued % np_}", issued // np_)
            issued += 1
        if gs < 0:
            continue
        for _ in range(kqps):
            if issued_b >= nb and mutant != "no_bempty_wait":
                yield ("wait", f"bempty{issued_b % nb}", issued_b // nb - 1)
            yield ("arrive", f"bfull{issued_b % nb}", issued_b // nb)
            yield ("copy", f"bfull{issued_b % nb}", issued_b // nb)
            issued_b += 1
            bunit += 1
            if bunit == qpt:
                bunit = 0
    # the mutant's extra quarters: a producer that believes a tile holds more B than it does
    if mutant == "quarters_per_tile_x_planes":
        for _ in range(qpt - g["NJ"] * 4):
            yield ("wait", f"bempty{issued_b % nb}", issued_b // nb - 1)
            issued_b += 1


def issuer(g, q):
    nb, naq, n_iss = C["kWNB"], g["NAQ"], C["kWIssuers"]
    Q = 0
    for lt in range(g["T"]):
        if lt > 0:
            yield ("wait", "dempty", lt - 1)
        for _ in range(g["NJ"] * 4):
            if Q % n_iss == q:
                yield ("wait", f"bfull{Q % nb}", Q // nb)
                yield ("wait", f"afull{Q % naq}", Q // naq)
                yield ("commit", q, f"aempty{Q % naq}", Q // naq)
                yield ("commit", q, f"bempty{Q % nb}", Q // nb)
            Q += 1
        yield ("commit", q, "dfull", lt)
    yield ("commit", q, "mma_done", 0)
    yield ("wait", "mma_done", 0)


def dequant(g, sub, mutant):
    np_, NAS, CPJ, CPQ = g["np"], g["NAS"], g["CPJ"], g["CPQ"]
    done0 = 0
    ps = 0
    for _ in range(g["T"]):
        for J in range(g["NJ"]):
            c0 = J * CPJ
            if c0 % 8 == 0:
                yield ("wait", f"pfull{ps % np_}", ps // np_)
            for cj in range(sub, CPJ, 2):
                cg = done0 + cj
                slot = (cg % NAS) // CPQ
                if cg >= NAS and mutant != "no_aempty_wait":
                    yield ("wait", f"aempty{slot}", cg // NAS - 1)
                yield ("arrive", f"afull{slot}", cg // NAS)
            done0 += CPJ
            if (c0 + CPJ) % 8 == 0:
                yield ("arrive", f"pempty{ps % np_}", ps // np_)
                ps += 1


def fold(g):
    # the fold warps move together (they meet at a named barrier every tile): one role, arriving
    # once per warp
    nf = C["kWFoldWarps"]
    for lt in range(g["T"]):
        yield ("wait", "dfull", lt)
        for _ in range(nf):
            yield ("arrive", "dempty", lt)
        if lt > 0:
            yield ("wait", "keys_free", lt - 1)
        for _ in range(nf):
            yield ("arrive", "keys_ready", lt)
        for _ in range(nf):  # their share of the selection jobs done
            yield ("arrive", "keys_free", lt)


def selection(g):
    ns = C["kWSelWarps"]
    for lt in range(g["T"]):
        yield ("wait", "keys_ready", lt)
        for _ in range(ns):
            yield ("arrive", "keys_free", lt)


def simulate(g, seed, mutant=None, max_steps=2_000_000):
    rng = random.Random(seed)
    nb, naq = C["kWNB"], g["NAQ"]
    bars = {}

    def add(name, count):
        bars[name] = Barrier(name, count)
    for i in range(g["np"]):
        add(f"pfull{i}", 2)                      # the producer's arrival + the copy's bytes
        add(f"pempty{i}", C["kWDeqWarps"])
    for i in range(nb):
        add(f"bfull{i}", 2)
        add(f"bempty{i}", 1)                     # the quarter's issuer
    for i in range(naq):
        add(f"afull{i}", 4 * g["CPQ"])           # the quadrant warps of the quarter's chunks
        add(f"aempty{i}", 1)
    add("dfull", C["kWIssuers"])
    add("dempty", C["kWFoldWarps"])
    add("mma_done", C["kWIssuers"])
    add("keys_ready", C["kWFoldWarps"])
    add("keys_free", C["kWSelWarps"] + C["kWFoldWarps"])

    roles = {"producer": producer(g, mutant), "fold": fold(g), "selection": selection(g)}
    for q in range(C["kWIssuers"]):
        roles[f"issuer{q}"] = issuer(g, q)
    for w in range(C["kWDeqWarps"]):
        roles[f"dequant{w}"] = dequant(g, w // 4, mutant)  # warps 0-3 even chunks, 4-7 odd
    nxt = {name: next(gen, None) for name, gen in roles.items()}
    copies = []                                   # (bar, phase), any order
    commits = {q: [] for q in range(C["kWIssuers"])}  # in order per issuing thread

    for _ in range(max_steps):
        options = []
        for name, act in nxt.items():
            if act is None:
                continue
            if act[0] == "wait" and not bars[act[1]].ready(act[2]):
                continue
            options.append(("role", name))
        options += [("copy", i) for i in range(len(copies))]
        options += [("commit", q) for q, lst in commits.items() if lst]
        if not options:
            if all(a is None for a in nxt.values()):
                return
            stuck = {n: a for n, a in nxt.items() if a is not None}
            raise Deadlock(f"stuck: {stuck}")
        kind, key = rng.choice(options)
        if kind == "copy":
            bar, ph = copies.pop(key)
            bars[bar].arrive(ph)
        elif kind == "commit":
            bar, ph = commits[key].pop(0)
            bars[bar].arrive(ph)
        else:
            act = nxt[key]
            if act[0] == "arrive":
                bars[act[1]].arrive(act[2])
            elif act[0] == "copy":
                copies.append((act[1], act[2]))
            elif act[0] == "commit":
                commits[act[1]].append((act[2], act[3]))
            nxt[key] = next(roles[key], None)
    raise AssertionError("step limit")


CONFIGS = [(G, ncol, K, tiles, np_)
           for G in (64, 128) for ncol in (32, 48, 64, 80) for K in (1024, 2048, 5120)
           for tiles, np_ in ((1, 3), (3, 4), (2, C["kWMaxNP"]))]


@pytest.mark.parametrize("G,NCOL,K,tiles,np_", CONFIGS)
def test_protocol_completes_without_aliasing(G, NCOL, K, tiles, np_):
    g = _geometry(G, NCOL, K, tiles, np_)
    for seed in range(5):
        simulate(g, seed)


@pytest.mark.parametrize("mutant,err", [
    ("quarters_per_tile_x_planes", Deadlock),  # the producer counts 16 units per group
    ("no_bempty_wait", Aliasing),               # B slots refilled before their issuer is done
    ("no_aempty_wait", Aliasing),               # A stages rewritten before their MMAs finish
])
def test_protocol_mutants_are_caught(mutant, err):
    g = _geometry(128, 80, 2048, 2, 4)
    with pytest.raises(err):
        for seed in range(5):
            simulate(g, seed, mutant)
