"""Progress of the fused decode kernel's schedule, checked on the CPU.

The decode kernel (csrc/decode_fused.cu) splits each CTA's work into a
sequence of chunks: every gate_up task's K chunks in task order, then the
down items. A producer warp's lane l issues chunks l, l + 32, ... into a ring
of kNS stages, chunk i once chunk i - kNS has been handed back; consumer
warps take chunks in sequence order by ticket. A gate_up chunk's stage is
handed back as soon as its words are read; its partial sums then wait for the
previous user of their buffer (task u - nb) to be finalised; the last of a
task's chunks finalises it and counts the expert's gate_up task done. A down
item holds its stage until all gate_up tasks of its expert, in every CTA,
are done.

This model plays that protocol for every CTA of a launch, in random order,
until nothing can move, and requires that every chunk of every CTA was
processed (no cycle of waits). The constants are read from the kernel source
so that the model follows it. Shapes include uneven K-chunk counts and the
largest H and E.
"""
import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "w4a16_mixture_experts_gb300", "csrc", "decode_fused.cu")


def _constants():
    src = open(SRC).read()
    c = {}
    for name in ("kCons", "kGC", "kGCMin", "kNS", "kRedMax", "kMaxNB", "kP2Rows"):
        m = re.search(r"constexpr int %s = (\d+);" % name, src)
        assert m, name
        c[name] = int(m.group(1))
    return c


C = _constants()


def _launch(T, H, E, k, I, nact, gc_max, sms=152):
    G1 = H // 128
    gc = min(G1, gc_max)
    nkc = -(-G1 // gc)
    nb = max(1, min(C["kMaxNB"], C["kRedMax"] // (nkc * 512)))
    tp1, tp2 = I // 8, H // C["kP2Rows"]
    n1, n2 = nact * tp1, nact * tp2
    chunks = min(T * k, E) * (tp1 * nkc + tp2)
    grid = max(1, min(sms, -(-chunks // C["kCons"])))
    return nkc, nb, tp1, tp2, n1, n2, grid


def _simulate(T, H, E, k, I, nact, seed, gc_max):
    rng = random.Random(seed)
    kCons, kNS = C["kCons"], C["kNS"]
    nkc, nb, tp1, tp2, n1, n2, grid = _launch(T, H, E, k, I, nact, gc_max)
    done1 = [0] * nact
    ctas = []
    for cb in range(grid):
        b1 = n1 * cb // grid
        m1 = n1 * (cb + 1) // grid - b1
        b2 = n2 * cb // grid
        m2 = n2 * (cb + 1) // grid - b2
        seq = [("gu", b1 + u, u) for u in range(m1) for _ in range(nkc)] + [("dn", b2 + d, 0) for d in range(m2)]
        ctas.append(dict(seq=seq, issued=set(), released=set(), ticket=0, held=[None] * kCons, cnt={}, fin=[0] * nb))
    moved = True
    while moved:
        moved = False
        for cta in ctas:
            seq = cta["seq"]
            for i in range(len(seq)):   # producer lanes
                if i in cta["issued"]:
                    continue
                if (i < 32 or i - 32 in cta["issued"]) and (i < kNS or i - kNS in cta["released"]):
                    cta["issued"].add(i)
                    moved = True
            for w in rng.sample(range(kCons), kCons):   # consumers
                st = cta["held"][w]
                if st is None:
                    if cta["ticket"] >= len(seq):
                        continue
                    st = cta["held"][w] = [cta["ticket"], "data"]
                    cta["ticket"] += 1
                    moved = True
                i, phase = st
                kind, task, u = seq[i]
                if phase == "data":
                    if i not in cta["issued"]:
                        continue
                    if kind == "dn":
                        if done1[task // tp2] < tp1:
                            continue
                        cta["released"].add(i)
                        cta["held"][w] = None
                        moved = True
                        continue
                    cta["released"].add(i)
                    st[1] = phase = "reduce"
                    moved = True
                if phase == "reduce":
                    b = u % nb
                    if cta["fin"][b] < u // nb:
                        continue
                    cta["cnt"][u] = cta["cnt"].get(u, 0) + 1
                    if cta["cnt"][u] == nkc:
                        cta["fin"][b] = u // nb + 1
                        done1[task // tp1] += 1
                    cta["held"][w] = None
                    moved = True
    stuck = [ci for ci, cta in enumerate(ctas)
             if cta["ticket"] < len(cta["seq"]) or any(h is not None for h in cta["held"])]
    return stuck, done1


@pytest.mark.parametrize("T,H,E,k,I,nact", [
    (1, 2560, 512, 10, 640, 10),
    (4, 2560, 512, 10, 640, 40),
    (7, 2560, 512, 10, 640, 70),
    (3, 1024, 1024, 32, 128, 95),
    (4, 256, 16, 2, 128, 8),
    (7, 3072, 64, 8, 256, 40),      # 5 or 6 K chunks per task, the last one shorter
    (2, 8064, 16, 4, 128, 8),       # 13 or 16 K chunks per task, 2 or 3 partial-sum buffers
    (7, 8064, 1024, 32, 640, 224),
])
def test_decode_schedule_completes(T, H, E, k, I, nact):
    # either chunk size the launch may choose (the larger unless its stages
    # leave no room for the activations)
    for gc_max in (C["kGC"], C["kGCMin"]):
        for seed in range(2):
            stuck, done1 = _simulate(T, H, E, k, I, nact, seed, gc_max)
            assert not stuck, "CTAs with chunks that can never be processed: %s" % stuck[:4]
            assert all(d == I // 8 for d in done1)
