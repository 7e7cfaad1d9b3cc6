"""The persistent grouped kernel's pipeline protocol, checked on the CPU.

Under QMM_GROUPED_PERSISTENT one CTA walks a list of output tiles ("items").
The weight ring, the activation ring and the tensor-memory A buffers run on
across items under one global group counter.  Each item's groups fill its
own ring stages, so an item's last stage may be short; the producer counts
the absent positions into that stage's release barrier when it issues it.
The accumulators go back and forth: the issuers' commit (acc_full) lets the
epilogue read them, and the epilogue's arrival (acc_empty) lets the next
item's MMAs write them.

This test runs a random-interleaving model of that protocol on the ring sizes
the launcher computes (`qmm_tc_persistent_pipeline_config`).  It checks four
things:
- every read sees the intended weight stage, activation stage and A buffer;
- no A buffer is rewritten before the MMA that reads it has completed;
- each epilogue sees, in each accumulator, exactly its item's groups;
- no item's MMA runs before every epilogue warp set has read the previous item.
A short stage lacks some consumers, which skip that lap of its slot.  The
parity waits stay sound because each consumer first passes the item's
accumulator hand-off, by which time every stage of the item has landed; the
model confirms it, and confirms that padding items to whole stages with
phantom groups (no copy, no MMA) is equally clean.  Two negative controls pin
the model itself: without the accumulator hand-back, or with A buffers shared
round-robin between dequantizer sets, it must report a violation.
"""
import random

import pytest

from split_w4a16_quantized_gb300 import build

GB300_SMEM_LIMIT = 232448 - 1040  # per-block opt-in maximum minus the kernel's call table


@pytest.fixture(scope="module")
def Q():
    build.build()
    from split_w4a16_quantized_gb300 import qmm
    return qmm


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, 0, 0

    def arrive(self, k=1):
        self.pending += k
        assert self.pending <= self.count, "more arrivals than the phase expects"
        if self.pending == self.count:
            self.pending = 0
            self.phase += 1

    def parity_done(self, parity):
        # mbarrier.try_wait.parity: has the phase with this parity completed?
        return (self.phase & 1) != parity


def layout(gpps, wgps, agps, pad):
    """Per global group position: (item, real, weight stage, activation stage),
    and the number of positions of every weight and activation stage.  Each
    item is cut into its own stages, the last one short (the kernel); with
    pad, it is first rounded up to whole weight stages with phantom groups."""
    pos, wsize, asize = [], [], []
    for r, gpp in enumerate(gpps):
        n = -(-gpp // wgps) * wgps if pad else gpp
        w0, a0 = len(wsize), len(asize)
        wsize += [min(wgps, n - k) for k in range(0, n, wgps)]
        asize += [min(agps, n - k) for k in range(0, n, agps)]
        for i in range(n):
            pos.append((r, i < gpp, w0 + i // wgps, a0 + i // agps))
    return pos, wsize, asize


def simulate(gpps, wgps, agps, nacc, sets, abuf, wst, ast, seed, pad=False, handoff=True,
             steps=400000):
    """One random interleaving; returns a list of violations (empty = clean)."""
    rng = random.Random(seed)
    pos, wsize, asize = layout(gpps, wgps, agps, pad)
    P, items = len(pos), len(gpps)
    w_full = [Barrier(1) for _ in range(wst)]
    w_empty = [Barrier(4 * wgps) for _ in range(wst)]
    act_full = [Barrier(1) for _ in range(ast)]
    act_empty = [Barrier(agps) for _ in range(ast)]
    a_full = [Barrier(4) for _ in range(abuf)]
    a_empty = [Barrier(1) for _ in range(abuf)]
    acc_full = Barrier(nacc)
    acc_empty = Barrier(sets)
    w_slot, act_slot, a_buf = [None] * wst, [None] * ast, [None] * abuf
    acc = [set() for _ in range(nacc)]          # groups summed into each accumulator
    acc_item = [None] * nacc
    mma_done = set()
    epi_done = [0] * items                      # sets whose epilogue of item r has read
    copies = []
    mma_queue = [[] for _ in range(nacc)]
    jw = ja = 0
    # each dequantizer set walks positions g = s, s + sets, ... and then,
    # after the last of an item, that item's epilogue
    set_seq = [[g for g in range(P) if g % sets == s] for s in range(sets)]
    set_k, set_step, set_item = [0] * sets, ["w"] * sets, [0] * sets
    iss_seq = [[g for g in range(P) if g % nacc == c] for c in range(nacc)]
    iss_k, iss_step, iss_item = [0] * nacc, ["start"] * nacc, [0] * nacc
    slow = rng.randrange(sets + nacc + 2)
    slow_p = rng.random() * 0.9
    bad = []

    def stalled(actor):
        return actor == slow and rng.random() < slow_p

    def real_groups(r, c):
        return {g for g, p in enumerate(pos) if p[0] == r and p[1] and g % nacc == c}

    for _ in range(steps):
        actors = []
        if jw < len(wsize) or ja < len(asize):
            actors.append(("producer",))
        actors += [("set", s) for s in range(sets) if set_item[s] < items]
        actors += [("issuer", c) for c in range(nacc) if iss_item[c] < items]
        if copies:
            actors.append(("copy",))
        if any(mma_queue):
            actors.append(("mma",))
        if not actors:
            break
        a = rng.choice(actors)
        if a[0] == "producer":
            if stalled(sets + nacc):
                continue
            if jw < len(wsize) and w_empty[jw % wst].parity_done(((jw // wst) & 1) ^ 1):
                if wsize[jw] < wgps:           # short stage: its absent positions count in
                    w_empty[jw % wst].arrive(4 * (wgps - wsize[jw]))
                copies.append(("w", jw % wst, jw))
                jw += 1
            if ja < len(asize) and act_empty[ja % ast].parity_done(((ja // ast) & 1) ^ 1):
                if asize[ja] < agps:
                    act_empty[ja % ast].arrive(agps - asize[ja])
                copies.append(("a", ja % ast, ja))
                ja += 1
        elif a[0] == "copy":       # copies land in any order
            ring, slot, stage = copies.pop(rng.randrange(len(copies)))
            if ring == "w":
                w_slot[slot] = stage
                w_full[slot].arrive()
            else:
                act_slot[slot] = stage
                act_full[slot].arrive()
        elif a[0] == "mma":        # one issuer's MMAs and commits complete in issue order
            c = rng.choice([c for c in range(nacc) if mma_queue[c]])
            if stalled(sets + nacc + 1) and len(mma_queue[c]) < 4:
                continue
            e = mma_queue[c].pop(0)
            if e[0] == "acc_full":
                acc_full.arrive()
                continue
            _, g, sa, ab, first, r = e
            if g is not None:                  # a real MMA writes accumulator c
                if r > 0 and epi_done[r - 1] < sets:
                    bad.append(("MMA before the previous epilogue read", g))
                if first:
                    acc[c], acc_item[c] = set(), r
                acc[c].add(g)
                mma_done.add(g)
            act_empty[sa].arrive()
            a_empty[ab].arrive()
        elif a[0] == "set":
            s = a[1]
            if stalled(s):
                continue
            r = set_item[s]
            if set_step[s] == "epi":
                if not acc_full.parity_done(r & 1):
                    continue
                for c in range(nacc):
                    want = real_groups(r, c)
                    if want and (acc_item[c] != r or acc[c] != want):
                        bad.append(("epilogue read of the wrong accumulator contents", r))
                epi_done[r] += 1
                if handoff:
                    acc_empty.arrive()
                set_item[s] += 1
                set_step[s] = "w"
                continue
            if set_k[s] >= len(set_seq[s]) or pos[set_seq[s][set_k[s]]][0] != r:
                set_step[s] = "epi"            # no positions left in item r
                continue
            g = set_seq[s][set_k[s]]
            _, real, j, _ = pos[g]
            ab = g % abuf
            if set_step[s] == "w":
                if not w_full[j % wst].parity_done((j // wst) & 1):
                    continue
                if w_slot[j % wst] != j:
                    bad.append(("weight read of the wrong stage", g))
                w_empty[j % wst].arrive(4)      # the set's four warps
                set_step[s] = "a"
            if set_step[s] == "a":
                if not a_empty[ab].parity_done(((g // abuf) & 1) ^ 1):
                    continue
                if real:
                    prev = g - abuf
                    if prev >= 0 and pos[prev][1] and prev not in mma_done:
                        bad.append(("A buffer overwritten before its MMA completed", g))
                    a_buf[ab] = g
                a_full[ab].arrive(4)
                set_k[s] += 1
                set_step[s] = "w"
        else:
            c = a[1]
            if stalled(sets + c):
                continue
            r = iss_item[c]
            if iss_step[c] == "start":
                if r > 0 and handoff and not acc_empty.parity_done((r - 1) & 1):
                    continue
                iss_step[c] = "act"
            if iss_k[c] >= len(iss_seq[c]) or pos[iss_seq[c][iss_k[c]]][0] != r:
                mma_queue[c].append(("acc_full",))   # the item's last commit
                iss_item[c] += 1
                iss_step[c] = "start"
                continue
            g = iss_seq[c][iss_k[c]]
            _, real, _, j = pos[g]
            ab = g % abuf
            if iss_step[c] == "act":
                if not act_full[j % ast].parity_done((j // ast) & 1):
                    continue
                if real and act_slot[j % ast] != j:
                    bad.append(("activation read of the wrong stage", g))
                iss_step[c] = "a"
            if iss_step[c] == "a":
                if not a_full[ab].parity_done((g // abuf) & 1):
                    continue
                if real and a_buf[ab] != g:
                    bad.append(("MMA read of the wrong A buffer contents", g))
                first = real and not any(pos[h][0] == r and pos[h][1] for h in iss_seq[c][:iss_k[c]])
                mma_queue[c].append(("mma", g if real else None, j % ast, ab, first, r))
                iss_k[c] += 1
                iss_step[c] = "act"
        if bad:
            return bad
    finished = all(x >= items for x in set_item) and all(x >= items for x in iss_item)
    return [] if finished else [("stalled", None)]


def _sweep(cfg, seeds, gpp_max, n_items=7, pad=False, handoff=True):
    failures = []
    for seed in range(seeds):
        rng = random.Random(1000 + seed)
        gpps = [rng.randint(1, gpp_max) for _ in range(n_items)]
        bad = simulate(gpps, cfg["weight_stage_groups"], cfg["act_stage_groups"],
                       cfg["issuers"], cfg["dequant_sets"], cfg["a_buffers"],
                       cfg["weight_stages"], cfg["act_stages"], seed, pad=pad,
                       handoff=handoff)
        if bad:
            failures.append((gpps, seed, bad[0]))
    return failures


@pytest.mark.parametrize("bm", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("gpp_max", [3, 10, 19])
def test_persistent_configurations_are_race_free(Q, bm, gpp_max):
    cfg = Q.qmm_tc_persistent_pipeline_config(bm, gpp_max, GB300_SMEM_LIMIT)
    assert cfg["smem"] <= GB300_SMEM_LIMIT
    assert cfg["a_buffers"] % cfg["dequant_sets"] == 0
    assert cfg["a_buffers"] % cfg["issuers"] == 0
    # full stages hold a group of every consumer
    assert cfg["weight_stage_groups"] >= cfg["dequant_sets"]
    assert (cfg["act_stage_groups"] >= cfg["issuers"] or
            cfg["act_stages"] % cfg["issuers"] == 0)
    failures = _sweep(cfg, seeds=12, gpp_max=gpp_max)
    assert not failures, (bm, cfg, failures[:3])


def test_padded_items_are_also_clean(Q):
    cfg = Q.qmm_tc_persistent_pipeline_config(32, 10, GB300_SMEM_LIMIT)
    assert not _sweep(cfg, seeds=12, gpp_max=10, pad=True)


def test_model_catches_a_missing_accumulator_handoff(Q):
    cfg = Q.qmm_tc_persistent_pipeline_config(32, 5, GB300_SMEM_LIMIT)
    assert _sweep(cfg, seeds=30, gpp_max=5, handoff=False)


def test_model_catches_a_buffers_shared_round_robin_across_items():
    # three dequantizer sets on four A buffers: a set's wait can take a
    # completion two laps old
    cfg = {"weight_stage_groups": 4, "act_stage_groups": 1, "issuers": 2, "dequant_sets": 3,
           "a_buffers": 4, "weight_stages": 3, "act_stages": 4}
    assert _sweep(cfg, seeds=40, gpp_max=12)
