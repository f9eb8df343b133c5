"""CPU model of the barrier protocol of the small-token INT4 kernel (moe_hm_gemm_gb300/csrc/
hm_gemm_f16s.cu): the producer, the issuing warps, the two dequant groups and the four epilogue
warps are generators of waits and arrivals over the kernel's mbarriers, run in random interleavings.
Every wait is evaluated twice: with the hardware's phase-parity rule (try_wait.parity sees the
phase with the given parity as complete) and with the exact number of phases the waiter means.
A disagreement means a waiter could be released by a phase two ahead of the one it wants (a
hazard); roles left waiting at the end are a deadlock. Test infrastructure, no GPU.

Each TMEM slot and its barriers belong to one (issuer, dequant group) pair, so each barrier has one
producer and one consumer in strict alternation; the model checks that property over the stream-K
and tile-parallel segment lists of the shapes the GPU tests run."""
import random

import pytest


def sk_start(c, total, g):
    return c * total // g


def segments(cta, tiles, kb_total, grid):
    """(tile, kb0, kb1) segments of one CTA's contiguous stream-K range."""
    total = tiles * kb_total
    it, end = sk_start(cta, total, grid), sk_start(cta + 1, total, grid)
    out = []
    while it < end:
        t, kb0 = divmod(it, kb_total)
        kb1 = min(kb0 + (end - it), kb_total)
        out.append((t, kb0, kb1))
        it += kb1 - kb0
    return out


class Hazard(Exception):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phases = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise Hazard(f"more arrivals than expected on {self.name}")
        if self.pending == 0:
            self.phases += 1
            self.pending = self.count

    def ready(self, parity, phases_needed):
        by_parity = (self.phases & 1) != parity
        exact = self.phases >= phases_needed
        if by_parity != exact:
            raise Hazard(f"{self.name}: parity {parity} reads {by_parity}, phase {phases_needed} reads {exact}")
        return by_parity


def build(segs, stages_ring, issuers, group=4, dq_group=4, empty_count=None):
    """Barriers and role generators for one CTA's segment list (group = 128-K blocks per load stage,
    dq_group = dequant warps per group). empty_count overrides the load-stage release count (a
    planted mistake for the negative control)."""
    bars = {}

    def bar(name, i, count):
        bars[(name, i)] = Barrier(f"{name}[{i}]", count)

    slots = 2 * issuers
    for s in range(stages_ring):
        bar("full_w", s, 1)
        bar("full_x", s, 1)
        bar("empty_l", s, empty_count if empty_count is not None else 4 + 2 * dq_group)
    for s in range(slots):
        bar("full_a", s, dq_group)
        bar("empty_a", s, 1)
        bar("acc_full", s, 1)
        bar("acc_empty", s, 4)
        bar("meta_full", 2 * s, dq_group)
        bar("meta_full", 2 * s + 1, dq_group)
    stages = []   # (segment, kb, blocks in stage, first block's sequence number, first pair number)
    seq = pair = 0
    for si, (_, a, b) in enumerate(segs):
        kb = a
        while kb < b:
            g = min(group, b - kb)
            stages.append((si, kb, g, seq, pair))
            seq += g
            pair += (g + 1) // 2
            kb += g

    def wait(key, parity, need):
        return ("wait", key, parity, need)

    def arrive(key, n=1):
        return ("arrive", key, n)

    def producer():
        for idx, _ in enumerate(stages):
            ls, n = idx % stages_ring, idx // stages_ring
            if idx >= stages_ring:
                yield wait(("empty_l", ls), (n & 1) ^ 1, n)
            yield arrive(("full_w", ls))
            yield arrive(("full_x", ls))

    def issuer(me):
        uses = [0, 0]
        for idx, (_, _, g, s0, p0) in enumerate(stages):
            ls, n = idx % stages_ring, idx // stages_ring
            have_x = False
            for j0 in range(0, g, 2):
                if (p0 + j0 // 2) % issuers != me:
                    continue
                if not have_x:
                    yield wait(("full_x", ls), n & 1, n + 1)
                    have_x = True
                nb = min(2, g - j0)
                for u in range(nb):
                    grp = (s0 + j0 + u) & 1
                    sl, k = 2 * me + grp, uses[grp]
                    yield wait(("acc_empty", sl), (k & 1) ^ 1, k)
                    yield wait(("full_a", sl), k & 1, k + 1)
                for u in range(nb):
                    grp = (s0 + j0 + u) & 1
                    sl = 2 * me + grp
                    yield arrive(("empty_a", sl))
                    yield arrive(("acc_full", sl))
                    uses[grp] += 1

    def dequant(grp):
        uses = [0] * issuers
        for idx, (_, _, g, s0, p0) in enumerate(stages):
            ls, n = idx % stages_ring, idx // stages_ring
            j0 = 0 if (s0 & 1) == grp else 1
            yield wait(("full_w", ls), n & 1, n + 1)
            if j0 >= g:
                yield arrive(("empty_l", ls))
            for jb in range(j0, g, 2):
                iss = (p0 + jb // 2) % issuers
                sl, k = 2 * iss + grp, uses[iss]
                yield wait(("empty_a", sl), (k & 1) ^ 1, k)
                yield arrive(("meta_full", 2 * sl + (k & 1)))
                if jb + 2 >= g:
                    yield arrive(("empty_l", ls))
                yield arrive(("full_a", sl))
                uses[iss] += 1

    def epilogue():
        uses = [0] * slots
        for idx, (_, _, g, s0, p0) in enumerate(stages):
            ls = idx % stages_ring
            for j in range(g):
                sl = 2 * ((p0 + j // 2) % issuers) + ((s0 + j) & 1)
                k = uses[sl]
                yield wait(("acc_full", sl), k & 1, k + 1)
                yield wait(("meta_full", 2 * sl + (k & 1)), (k >> 1) & 1, (k >> 1) + 1)
                yield arrive(("acc_empty", sl))
                uses[sl] += 1
            yield arrive(("empty_l", ls))

    roles = {"producer": producer()}
    for i in range(issuers):
        roles[f"issuer{i}"] = issuer(i)
    for grp in range(2):
        for w in range(dq_group):
            roles[f"dequant{grp}.{w}"] = dequant(grp)
    for q in range(4):
        roles[f"epilogue{q}"] = epilogue()
    return bars, roles


def run(bars, roles, rng):
    """Random interleaving to the end; returns the roles left waiting (empty = finished)."""
    cur = {k: next(v, None) for k, v in roles.items()}
    while True:
        ready = [k for k, op in cur.items()
                 if op is not None and (op[0] == "arrive" or bars[op[1]].ready(op[2], op[3]))]
        if not ready:
            return {k: op for k, op in cur.items() if op is not None}
        k = rng.choice(ready)
        op = cur[k]
        if op[0] == "arrive":
            bars[op[1]].arrive(op[2])
        cur[k] = next(roles[k], None)


SHAPES = [(4096, 4096), (14336, 4096), (4096, 14336), (640, 3072), (256, 1024), (384, 14336), (512, 2048)]


@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("m", [1, 9, 16, 17, 32])
def test_no_hazard_or_deadlock(n, k, m):
    bt = 16 if m <= 16 else 32
    ring, issuers = (4, 3) if bt == 16 else (3, 2)       # load stages and issuing warps of the kernel
    tiles, kb_total = (n // 128) * ((m + bt - 1) // bt), k // 128
    rng = random.Random(n * 131 + k * 7 + m)
    for stream_k in (True, False):
        grid = min(152, tiles * kb_total) if stream_k else min(152, tiles)
        for cta in rng.sample(range(grid), min(grid, 6)):
            segs = segments(cta, tiles, kb_total, grid) if stream_k else [(t, 0, kb_total) for t in range(cta, tiles, grid)]
            bars, roles = build(segs, ring, issuers)
            left = run(bars, roles, rng)
            assert not left, f"deadlock: n={n} k={k} m={m} stream_k={stream_k} cta={cta}: {left}"


def test_model_flags_a_planted_mistake():
    """Negative control: a load-stage release barrier that expects one arrival more than its roles
    make never completes, and the model reports the producer stuck on it."""
    segs = segments(0, 32, 32, 8)            # 128 k-blocks: the ring of 4 load stages turns over
    bars, roles = build(segs, 4, 3, empty_count=4 + 2 * 4 + 1)
    left = run(bars, roles, random.Random(0))
    assert "producer" in left and left["producer"][1][0] == "empty_l"
