"""Progress of the fused decode kernel's schedule, checked on the CPU.

The decode kernel (csrc/decode_fused.cu) splits each CTA's work into a
sequence of chunks: every gate_up task's K chunks in task order, then the
down chunks of the output blocks it owns (block by block, one chunk per active
expert). A producer warp's lane l issues chunks l, l + 32, ... into a ring of
kNS stages, chunk i once chunk i - kNS has been handed back; consumer warps
take chunks in sequence order by ticket. A gate_up chunk's stage is handed
back as soon as its words are read; its partial sums then wait for the
previous user of their buffer (task u - nb) to be finalised; the last of a
task's chunks finalises it and counts the expert's gate_up task done. A down
chunk holds its stage until all gate_up tasks of its expert, in every CTA,
are done, (when its block buffer lives in the partial-sum area) until every
gate_up task of its own CTA is finalised, and until the block that used its
buffer before is combined; the chunk that completes a block combines it.

This model plays that protocol for every CTA of a launch, in random order,
until nothing can move, and requires that every chunk of every CTA was
processed (no cycle of waits). The constants are read from the kernel source
so that the model follows it. Shapes include uneven K-chunk counts and the
largest H and E.
"""
import math
import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "w4a16_mixture_experts_gb300", "csrc", "decode_fused.cu")


def _constants():
    src = open(SRC).read()
    c = {}
    for name in ("kFW", "kCons", "kGC", "kGCMin", "kNS", "kRedMax", "kMaxNB", "kP2Rows", "kDecodeMaxT",
                 "kFastN", "kRingWordsExtra", "kSpreadDownWeight"):
        m = re.search(r"constexpr int %s = (\d+);" % name, src)
        assert m, name
        c[name] = int(m.group(1))
    m = re.search(r"constexpr int kFusedSmem = (\d+) - (\d+);", src)
    assert m, "kFusedSmem"
    c["kFusedSmem"] = int(m.group(1)) - int(m.group(2))
    return c


C = _constants()


def _al(v, a):
    return (v + a - 1) // a * a


def _layout_gc(T, H, E, k, I, gc_max, full=False):
    """Mirror of fused_layout_gc: (fits, staged activations, gcw); with full, also
    (output-block buffers, whether they have a region of their own)."""
    G1, G2 = H // 128, I // 128
    gc = min(G1, gc_max)
    gcw = gc * 16
    nkc = -(-G1 // gc)
    p1 = 2 * 8 * gcw * 4
    p2 = C["kP2Rows"] * (I // 2)
    stage = _al(max(p1, p2), 128)
    nb = max(1, min(C["kMaxNB"], C["kRedMax"] // (nkc * 512)))
    red_off = C["kNS"] * stage
    yb = T * k * C["kP2Rows"] * 4
    area = max(nb * nkc * 512, yb)
    red = area + 2 * nb * 4 + 4 + 2 * C["kNS"] * 4 + 4 * C["kRingWordsExtra"]
    nyb = min(2, area // yb) if yb else 0
    pro_off = red_off + _al(red, 128)
    n = T * k
    na = max(1, min(E, n))
    pro = (_al(n * 2, 16) * 3 + _al(C["kFastN"] * 4, 16) + _al(na * 2, 16) * 3 + _al(T * 2, 16) + 4 * C["kFW"] * 8
           + 16 + _al(n * 4, 16))
    xs = T * H * 2 + _al(T * G1 * 4, 16)
    base = pro_off + _al(pro, 128)
    staged = base + xs <= C["kFusedSmem"]
    total = base + xs if staged else base
    ys_start = _al(total, 128)
    ysep = bool(yb) and ys_start + 2 * yb <= C["kFusedSmem"]
    if ysep:
        nyb, total = 2, ys_start + 2 * yb
    ok = total <= C["kFusedSmem"] and T <= C["kDecodeMaxT"] and k <= 32 and I <= 1280 and gcw <= 256 and \
        (nyb >= 1 or T == 0)
    return (ok, staged, gcw, nyb, ysep, red_off) if full else (ok, staged, gcw)


def _route_scratch_start():
    m = re.search(r"constexpr uint32_t kRtLogit = (\d+);", open(SRC).read())
    assert m, "kRtLogit"
    return int(m.group(1))


def _route_max_t():
    m = re.search(r"constexpr int kRouteFusedMaxT = (\d+);", open(SRC).read())
    assert m, "kRouteFusedMaxT"
    return int(m.group(1))


def fused_plan(T, H, E, k, I):
    """Mirror of fused_layout: None if the decode kernel cannot take the shape,
    else (staged, groups per chunk, separate block buffers, routes itself):
    which instantiation of the kernel runs, which of its two buffer
    placements, and whether the router's scratch (the logits after a fixed
    head) fits the ring, which it occupies before the first weight copy."""
    a = _layout_gc(T, H, E, k, I, C["kGC"], full=True)
    if not (a[0] and a[1]):
        b = _layout_gc(T, H, E, k, I, C["kGCMin"], full=True)
        a = b if b[0] and (b[1] or not a[0]) else a
    if not a[0]:
        return None
    route = a[1] and T <= _route_max_t() and T * k <= C["kFastN"] and _route_scratch_start() + 4 * T * E <= a[5]
    return a[1], a[2] // 16, a[4], route


def _launch(T, H, E, k, I, nact, gc_max, sms=152):
    G1 = H // 128
    gc = min(G1, gc_max)
    nkc = -(-G1 // gc)
    nb = max(1, min(C["kMaxNB"], C["kRedMax"] // (nkc * 512)))
    _, _, _, nyb, ysep, _ = _layout_gc(T, H, E, k, I, gc_max, full=True)
    tp1 = I // 8
    n1 = nact * tp1
    chunks = min(T * k, E) * (tp1 * nkc + H // C["kP2Rows"])
    grid = max(1, min(sms, -(-chunks // C["kCons"])))
    # the kernel instantiation with the spread task order and its split weight
    spread = min(T * k, E) * tp1 * nkc > 2 * C["kCons"] * grid
    return nkc, nb, nyb, ysep, tp1, n1, grid, spread


def _split(H, I, nact, Cg, cb, w=1):
    """Mirror of fused_split and its host constants: (first gate_up task, tasks,
    first block, end block); w weighs a CTA's own down bytes. The task bounds
    are f(c) = floor(n1 * (fp32(cum(c)) * fp32(1 / cum(Cg)))), in fp32 as the
    kernel computes them."""
    import numpy as np
    B = H // C["kP2Rows"]
    n1 = nact * (I // 8)
    cb0, cb1 = B * cb // Cg, B * (cb + 1) // Cg
    bmin = B // Cg
    unit = (I // 8) * H + B * I
    x0 = max(0, unit - Cg * w * I * bmin)
    x1 = max(0, unit - Cg * w * I * (bmin + 1))
    allv = Cg * x0 + (B - bmin * Cg) * (x1 - x0)
    r = np.float32(1.0 / allv) if allv > 0 else np.float32(0.0)

    def at(c):
        if c <= 0:
            return 0
        if c >= Cg:
            return n1
        if r == 0:
            return n1 * c // Cg
        nbig = B * c // Cg - bmin * c
        cum = c * x0 + nbig * (x1 - x0)
        return int(np.floor(np.float32(n1) * (np.float32(cum) * r)))

    s0, s1 = at(cb), at(cb + 1)
    return s0, s1 - s0, cb0, cb1


def task_stride(n1, nkc, grid):
    """Mirror of task_stride: 0, or the multiplier M of the global task order."""
    if n1 * nkc <= 2 * C["kCons"] * grid:
        return 0
    M = max(1, (n1 * 633) >> 10)
    while math.gcd(M, n1) != 1:
        M += 1
    return M


def cta_tasks(b1, m1, n1, M):
    """The CTA's gate_up tasks in the order it takes them."""
    if M == 0 or m1 > C["kFW"] * 32:
        return list(range(b1, b1 + m1)) if M == 0 else [(x * M) % n1 for x in range(b1, b1 + m1)]
    return sorted((x * M) % n1 for x in range(b1, b1 + m1))


def _simulate(T, H, E, k, I, nact, seed, gc_max):
    rng = random.Random(seed)
    kCons, kNS = C["kCons"], C["kNS"]
    nkc, nb, nyb, ysep, tp1, n1, grid, spread = _launch(T, H, E, k, I, nact, gc_max)
    M = task_stride(n1, nkc, grid) if spread else 0
    w = C["kSpreadDownWeight"] if M else 1
    done1 = [0] * nact
    ctas = []
    covered_tasks, covered_blocks = [], []
    for cb in range(grid):
        b1, m1, cb0, cb1 = _split(H, I, nact, grid, cb, w)
        tasks = cta_tasks(b1, m1, n1, M)
        covered_tasks += tasks
        covered_blocks += list(range(cb0, cb1))
        # down chunks block by block, or (spread order) expert by expert when every block has a buffer
        if M and cb1 - cb0 <= nyb:
            down = [("dn", a, c - cb0) for a in range(nact) for c in range(cb0, cb1)]
        else:
            down = [("dn", a, c - cb0) for c in range(cb0, cb1) for a in range(nact)]
        seq = [("gu", tasks[u], u) for u in range(m1) for _ in range(nkc)] + down
        ctas.append(dict(seq=seq, issued=set(), released=set(), ticket=0, held=[None] * kCons, cnt={}, fin=[0] * nb,
                         m1=m1, gu_done=0, dcnt=[0] * nyb, dfin=[0] * nyb))
    # the split covers every gate_up task and every output block exactly once
    assert sorted(covered_tasks) == list(range(n1))
    assert sorted(covered_blocks) == list(range(H // C["kP2Rows"]))
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
                        a, lb = task, u
                        buf = lb % nyb
                        if done1[a] < tp1 or (not ysep and cta["gu_done"] < cta["m1"]) or \
                                cta["dfin"][buf] < lb // nyb:
                            continue
                        cta["dcnt"][buf] += 1
                        if cta["dcnt"][buf] == nact:
                            cta["dcnt"][buf] = 0
                            cta["dfin"][buf] = lb // nyb + 1
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
                        cta["gu_done"] += 1
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
    (7, 4096, 8, 8, 128, 8),        # block buffers in the partial-sum area
])
def test_decode_schedule_completes(T, H, E, k, I, nact):
    # either chunk size the launch may choose (the larger unless its stages
    # leave no room for the activations)
    for gc_max in (C["kGC"], C["kGCMin"]):
        for seed in range(2):
            stuck, done1 = _simulate(T, H, E, k, I, nact, seed, gc_max)
            assert not stuck, "CTAs with chunks that can never be processed: %s" % stuck[:4]
            assert all(d == I // 8 for d in done1)


# The shapes of the GPU parity tests that run the decode kernel, and the
# instantiation each one reaches: decode_fused_kernel<true, *> stages the
# activations in shared memory, <false, *> reads them from global memory.
# GPU_SHARED_AREA_SHAPES lists those whose down outputs' block buffers reuse
# the gate_up partial-sum area (all others have a region of their own).
GPU_SHARED_AREA_SHAPES = {(7, 4096, 8, 8, 128)}
GPU_DECODE_SHAPES = {
    (7, 4096, 8, 8, 128): True,        # block buffers in the partial-sum area
    (1, 2560, 512, 10, 640): True,     # decode1
    (4, 2560, 512, 10, 640): True,     # decode4
    (4, 256, 16, 2, 128): True,        # tiny
    (7, 2560, 512, 10, 640): True,     # the largest decode batch at full shape
    (1, 128, 1, 1, 128): True,
    (5, 384, 24, 3, 256): True,
    (3, 1024, 1024, 32, 128): True,
    (7, 3072, 64, 8, 256): True,
    (2, 8064, 16, 4, 128): True,
    (3, 128, 1024, 32, 128): True,     # E and k at their maxima, the smallest H
    (7, 8064, 64, 8, 128): False,      # x too large to stage next to the ring
    (7, 7168, 32, 4, 256): False,
    (6, 6144, 32, 4, 256): True,       # staged with 4-group chunks
}


@pytest.mark.parametrize("shape,staged", sorted(GPU_DECODE_SHAPES.items()))
def test_decode_instantiation_of_gpu_shapes(shape, staged):
    plan = fused_plan(*shape)
    assert plan is not None, "the decode kernel must take %s" % (shape,)
    assert plan[0] == staged
    assert plan[2] == (shape not in GPU_SHARED_AREA_SHAPES)
    if shape == (6, 6144, 32, 4, 256):
        assert plan[1] == C["kGCMin"]
    # the library's own choice (a host-only query) agrees with this mirror
    assert _library_plan(*shape) == plan


def _library_plan(*dims):
    import w4a16_mixture_experts_gb300 as moe
    moe.build()
    return moe.moe_forward_plan(*dims)


def test_mirror_matches_library_plan_over_many_shapes():
    import itertools
    for T, H, E, k, I in itertools.product((1, 3, 7, 8), (128, 2560, 6144, 8064), (16, 512, 1024),
                                           (1, 10, 32), (128, 640, 1280, 1408)):
        if k > E:
            continue
        assert _library_plan(T, H, E, k, I) == fused_plan(T, H, E, k, I), (T, H, E, k, I)
    # shapes whose block buffers stay in the partial-sum area
    for shape in ((7, 4096, 8, 8, 128), (6, 4608, 8, 8, 128), (5, 5888, 8, 4, 128), (4, 7296, 8, 8, 128)):
        assert fused_plan(*shape)[2] is False
        assert _library_plan(*shape) == fused_plan(*shape), shape


def test_router_runs_inside_the_decode_kernel_at_the_benchmark_shapes():
    # the full layer shape (with and without the shared expert) up to the
    # kernel's batch limit for it, and the largest router there (1024 experts)
    tmax = _route_max_t()
    for T in range(1, C["kDecodeMaxT"] + 1):
        assert fused_plan(T, 2560, 512, 10, 640)[3] == (T <= tmax), T
        assert fused_plan(T, 2560, 513, 11, 640)[3] == (T <= tmax), T
    assert fused_plan(tmax, 2560, 1024, 32, 640)[3]
    # the smallest ring (H = I = 128) still holds the logits of tmax tokens x 1024 experts
    assert fused_plan(tmax, 128, 1024, 8, 128)[3]
    assert not fused_plan(tmax + 1, 2560, 512, 10, 640)[3]


def test_decode_takes_every_batch_up_to_its_limit_at_full_shape():
    for T in range(1, C["kDecodeMaxT"] + 1):
        for k in (1, 10, 32):
            for E in (k, 512, 1024):
                assert fused_plan(T, 2560, E, k, 640) is not None, (T, E, k)
    assert fused_plan(C["kDecodeMaxT"] + 1, 2560, 512, 10, 640) is None


def _warp_prologue(ids):
    """Mirror of f_route_prologue's warp: bitonic sort of (expert << 5 | a) over 32
    lanes by xor-shuffles, then the slots and the runs of equal experts."""
    n = len(ids)
    key = [(ids[l] << 5) | l if l < n else 0x7fffffff for l in range(32)]
    kk = 2
    while kk <= 32:
        j = kk >> 1
        while j > 0:
            o = [key[l ^ j] for l in range(32)]
            key = [min(key[l], o[l]) if ((l & j) == 0) == ((l & kk) == 0) else max(key[l], o[l]) for l in range(32)]
            j >>= 1
        kk <<= 1
    e = [k >> 5 for k in key]
    a = [k & 31 for k in key]
    starts = [l < n and (l == 0 or e[l - 1] != e[l]) for l in range(32)]
    perm = a[:n]
    inv = [0] * n
    for s in range(n):
        inv[a[s]] = s
    act, aoff, acnt = [], [], []
    pos = [l for l in range(32) if starts[l]]
    for i, l in enumerate(pos):
        act.append(e[l])
        aoff.append(l)
        acnt.append((pos[i + 1] if i + 1 < len(pos) else n) - l)
    return perm, inv, act, aoff, acnt


def test_route_prologue_network_matches_the_ranking():
    # the general prologue's definition: slot = #ids below e + #earlier equal ids;
    # the active list in increasing expert order with first slot and count
    rng = random.Random(7)
    for trial in range(300):
        T = rng.choice([1, 2])
        k = rng.randint(1, 32 // T)
        E = rng.choice([k, max(k, 16), 64, 512, 1024])
        ids = []
        for t in range(T):
            ids += rng.sample(range(E), k)   # distinct within a token, repeats across tokens
        n = len(ids)
        perm, inv, act, aoff, acnt = _warp_prologue(ids)
        for a in range(n):
            slot = sum(1 for x in ids if x < ids[a]) + sum(1 for b in range(a) if ids[b] == ids[a])
            assert inv[a] == slot and perm[slot] == a, (trial, ids)
        assert act == sorted(set(ids))
        assert aoff == [sum(1 for x in ids if x < e) for e in act]
        assert acnt == [ids.count(e) for e in act]
