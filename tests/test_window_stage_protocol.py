"""Host model of the draft-window kernel's stage protocol (CPU only).

attn_window_bf16 streams a segment's 64-key tiles through 3 shared-memory stages (tile t in
stage t % 3); two groups of four warps take alternate tiles (group t % 2); the last warp of a
group to finish a tile re-issues the stage's copy for tile t + 3; consumers wait for a tile with
an mbarrier parity wait.  A parity wait passes as soon as the barrier's current phase has the
other parity, so it is only sound if the waiter can never be two phases behind.  This model plays
the protocol under random copy and compute latencies and checks every wait that passes against
the phase it wanted:

* the kernel's form (one full barrier per (group, stage), tile t completing phase t // 6 of
  barrier (t % 2, t % 3)) never passes early and never stalls;
* the form with one barrier per stage (phase t // 3 of barrier t % 3), in which a group skips the
  other group's phases, does pass early in some schedules -- the model can see the failure it
  guards against.
"""

import random

STAGES, GROUPS, WARPS_PER_GROUP = 3, 2, 4


def play(ntiles: int, per_group: bool, seed: int) -> str:
    rnd = random.Random(seed)
    bar = (lambda t: (t % GROUPS) * STAGES + t % STAGES) if per_group else (lambda t: t % STAGES)
    phase = (lambda t: t // (GROUPS * STAGES)) if per_group else (lambda t: t // STAGES)
    completed = [0] * (GROUPS * STAGES)   # completed phases per barrier
    in_stage = {}                         # stage -> tile whose copy was issued last
    landing = {}                          # tile -> time its copy completes
    now = 0.0
    for t in range(min(STAGES, ntiles)):  # the first copies, issued up front
        landing[t] = rnd.uniform(1.0, 3.0)
        in_stage[t % STAGES] = t
    finished = [0] * STAGES               # warp-tiles finished per stage (never reset)
    warps = [dict(next=w // WARPS_PER_GROUP, busy=0.0, tile=None) for w in range(GROUPS * WARPS_PER_GROUP)]
    consumed = 0
    for _ in range(200000):
        for t, at in list(landing.items()):
            if at <= now:
                completed[bar(t)] += 1
                del landing[t]
        for w in warps:                   # waits
            t = w["next"]
            if t >= ntiles or w["tile"] is not None:
                continue
            k = phase(t)
            if (completed[bar(t)] & 1) != (k & 1):          # the parity wait passes
                if completed[bar(t)] != k + 1 or in_stage.get(t % STAGES) != t:
                    return "early"
                w["tile"], w["busy"], w["next"] = t, now + rnd.uniform(0.5, 2.5), t + GROUPS
        for w in warps:                   # finished tiles: the group's last warp refills the stage
            if w["tile"] is not None and w["busy"] <= now:
                t, w["tile"] = w["tile"], None
                s = t % STAGES
                finished[s] += 1
                if finished[s] % WARPS_PER_GROUP == 0:
                    consumed += 1
                    if t + STAGES < ntiles:
                        in_stage[s] = t + STAGES
                        landing[t + STAGES] = now + rnd.uniform(1.0, 3.0)
        if consumed == ntiles:
            return "ok"
        future = [x for x in landing.values()] + [w["busy"] for w in warps if w["tile"] is not None]
        if not future:
            return "stalled"
        now = max(now, min(future))
    return "stalled"


def test_per_group_barriers_never_pass_early():
    for ntiles in (1, 2, 3, 4, 8, 16, 40):
        for seed in range(150):
            assert play(ntiles, True, seed) == "ok", (ntiles, seed)


def test_shared_barriers_can_pass_early():
    outcomes = {play(ntiles, False, seed) for ntiles in (8, 16, 40) for seed in range(150)}
    assert "early" in outcomes
