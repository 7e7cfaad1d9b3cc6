"""The tcgen05 W4A16 kernel's pipeline protocol, checked on the CPU.

The kernel moves every 128-group through four mbarrier rings:
- the weight ring (producer -> dequantizer sets);
- the activation ring (producer -> MMA issuers);
- the tensor-memory A buffers (dequantizer sets -> issuers, released by the
  issuers' MMA commits);
- the accumulators.
Every wait is a phase-parity wait.  A parity wait is sound only if the waiter
also waited on the previous lap of the same slot; otherwise a completion two
laps old satisfies it.  The kernel sizes its rings to keep that true.

This test runs a random-interleaving model of exactly that protocol on the
configurations the kernel uses (`qmm_tc_pipeline_config`, the launcher's own
computation).  TMA copies land in any order, and each issuer's MMAs complete
in issue order.  The model checks that every read sees the intended data and
that no A buffer is overwritten before the MMA that reads it has completed.
Two layouts known to be unsafe must be caught, so the model itself is pinned.
"""
import random

import pytest

from split_w4a16_quantized_gb300 import build

GB300_SMEM_LIMIT = 232448 - 16  # per-block opt-in maximum minus static shared memory


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


def simulate(gpp, wgps, agps, nacc, sets, abuf, wst, ast, seed, steps=400000):
    """One random interleaving; returns a list of violations (empty = clean)."""
    rng = random.Random(seed)
    nw, na = -(-gpp // wgps), -(-gpp // agps)
    w_full = [Barrier(1) for _ in range(wst)]
    w_empty = [Barrier(4 * wgps) for _ in range(wst)]
    act_full = [Barrier(1) for _ in range(ast)]
    act_empty = [Barrier(agps) for _ in range(ast)]
    a_full = [Barrier(4) for _ in range(abuf)]
    a_empty = [Barrier(1) for _ in range(abuf)]
    w_slot, act_slot, a_buf = [None] * wst, [None] * ast, [None] * abuf
    mma_done = set()
    copies = []                      # (ring, slot, stage) copies in flight
    mma_queue = [[] for _ in range(nacc)]
    jw = ja = 0
    set_pos, set_step = list(range(sets)), ["w"] * sets
    iss_pos, iss_step = list(range(nacc)), ["act"] * nacc
    slow = rng.randrange(sets + nacc + 2)
    slow_p = rng.random() * 0.9
    bad = []

    def stalled(actor):
        return actor == slow and rng.random() < slow_p

    for _ in range(steps):
        actors = []
        if jw < nw or ja < na:
            actors.append(("producer",))
        actors += [("set", s) for s in range(sets) if set_pos[s] < gpp]
        actors += [("issuer", c) for c in range(nacc) if iss_pos[c] < gpp]
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
            if jw < nw and w_empty[jw % wst].parity_done(((jw // wst) & 1) ^ 1):
                copies.append(("w", jw % wst, jw))
                jw += 1
            if ja < na and act_empty[ja % ast].parity_done(((ja // ast) & 1) ^ 1):
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
        elif a[0] == "mma":        # one issuer's MMAs complete in issue order
            c = rng.choice([c for c in range(nacc) if mma_queue[c]])
            if stalled(sets + nacc + 1) and len(mma_queue[c]) < 4:
                continue
            i, sa, ab = mma_queue[c].pop(0)
            mma_done.add(i)
            act_empty[sa].arrive()
            a_empty[ab].arrive()
        elif a[0] == "set":
            s = a[1]
            if stalled(s):
                continue
            i = set_pos[s]
            j, ab = i // wgps, i % abuf
            if set_step[s] == "w":
                if not w_full[j % wst].parity_done((j // wst) & 1):
                    continue
                if w_slot[j % wst] != j:
                    bad.append(("weight read of the wrong stage", i))
                w_empty[j % wst].arrive(4)      # the set's four warps
                set_step[s] = "a"
            if set_step[s] == "a":
                if not a_empty[ab].parity_done(((i // abuf) & 1) ^ 1):
                    continue
                if i >= abuf and (i - abuf) not in mma_done:
                    bad.append(("A buffer overwritten before its MMA completed", i))
                a_buf[ab] = i
                a_full[ab].arrive(4)
                set_pos[s] += sets
                set_step[s] = "w"
        else:
            c = a[1]
            if stalled(sets + c):
                continue
            i = iss_pos[c]
            j, ab = i // agps, i % abuf
            if iss_step[c] == "act":
                if not act_full[j % ast].parity_done((j // ast) & 1):
                    continue
                if act_slot[j % ast] != j:
                    bad.append(("activation read of the wrong stage", i))
                iss_step[c] = "a"
            if iss_step[c] == "a":
                if not a_full[ab].parity_done((i // abuf) & 1):
                    continue
                if a_buf[ab] != i:
                    bad.append(("MMA read of the wrong A buffer contents", i))
                mma_queue[c].append((i, j % ast, ab))
                iss_pos[c] += nacc
                iss_step[c] = "act"
        if bad:
            return bad
    finished = all(p >= gpp for p in set_pos) and all(p >= gpp for p in iss_pos)
    return [] if finished else [("stalled", None)]


def _sweep(cfg, gpps, seeds):
    failures = []
    for gpp in gpps:
        for seed in range(seeds):
            bad = simulate(gpp, cfg["weight_stage_groups"], cfg["act_stage_groups"],
                           cfg["issuers"], cfg["dequant_sets"], cfg["a_buffers"],
                           cfg["weight_stages"], cfg["act_stages"], seed)
            if bad:
                failures.append((gpp, seed, bad[0]))
    return failures


@pytest.mark.parametrize("bm", [16, 32, 64, 128, 256])
def test_kernel_configurations_are_race_free(Q, bm):
    for gpp in (1, 2, 3, 5, 10, 19, 38):
        cfg = Q.qmm_tc_pipeline_config(bm, gpp, GB300_SMEM_LIMIT)
        # the sizing rules themselves
        assert cfg["a_buffers"] % cfg["dequant_sets"] == 0
        assert cfg["a_buffers"] % cfg["issuers"] == 0
        assert (cfg["weight_stage_groups"] >= cfg["dequant_sets"] or
                cfg["weight_stages"] * cfg["weight_stage_groups"] % cfg["dequant_sets"] == 0)
        assert (cfg["act_stage_groups"] >= cfg["issuers"] or
                cfg["act_stages"] * cfg["act_stage_groups"] % cfg["issuers"] == 0)
        assert cfg["smem"] <= GB300_SMEM_LIMIT
        failures = _sweep(cfg, [gpp], seeds=25)
        assert not failures, (bm, cfg, failures[:3])


def test_model_catches_a_buffers_shared_round_robin():
    # three dequantizer sets on four A buffers: a set's wait can take a
    # completion two laps old (the race an earlier kernel version had)
    cfg = {"weight_stage_groups": 4, "act_stage_groups": 1, "issuers": 2, "dequant_sets": 3,
           "a_buffers": 4, "weight_stages": 3, "act_stages": 4}
    assert _sweep(cfg, [19, 38], seeds=40)


def test_model_catches_an_activation_ring_that_skips_a_lap():
    # two issuers on an odd activation ring of one-group stages: an issuer
    # waits on a slot whose previous lap belonged to the other issuer
    cfg = {"weight_stage_groups": 4, "act_stage_groups": 1, "issuers": 2, "dequant_sets": 2,
           "a_buffers": 4, "weight_stages": 3, "act_stages": 3}
    assert _sweep(cfg, [19, 38], seeds=40)


def test_configuration_query_rejects_bad_arguments(Q):
    with pytest.raises(Q.QmmError):
        Q.qmm_tc_pipeline_config(48, 4)
    with pytest.raises(Q.QmmError):
        Q.qmm_tc_pipeline_config(32, 0)
    with pytest.raises(Q.QmmError):       # nothing fits in 64 KB
        Q.qmm_tc_pipeline_config(128, 4, 64 * 1024)
