"""CPU model of the block-scaled CTA-pair GEMM's stage protocol (csrc/gemm.cu), checked under random
schedules.

Roles: two TMA producers (one per CTA), eight scale writers (four per CTA), the MMA issuer, and the
tensor core completing the MMAs of each stage step in order.  Operand stages form a ring of
kBsPairStages `full` / `empty` mbarriers; each stage step's E8M0 scales go to TMEM slots that form a
ring of kSfRing steps.  A producer refills stage s once step s - kBsPairStages is complete; a writer
writes step s's slots once step s - kSfAhead is complete, kSfAhead = min(kSfRing, kBsPairStages); the
issuer waits for `full[s]` (both producers and all writers); each completion arrives on `empty[s]`.

The model keeps each mbarrier's phase count and checks what the hardware does not: a phase never
receives more arrivals than its count, a parity wait never waits on a phase two or more completions
old (it would see the wrong parity), the MMAs of a step read the scales written for that step, and
no schedule deadlocks.  The constants are read from the kernel source, so a change to the ring sizes
is checked too."""
import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GEMM = os.path.join(ROOT, "scaling_quantization_gemm_gb300", "csrc", "gemm.cu")


def _const(src, name):
    m = re.search(r"constexpr int %s = (\d+);" % name, src)
    assert m, name
    return int(m.group(1))


def kernel_constants():
    src = open(GEMM).read()
    bn, accs = _const(src, "kBnPair"), _const(src, "kAccBufs")
    cols, kps, stages = _const(src, "kSfColsPerStage"), _const(src, "kBsKPerStage"), _const(src, "kBsPairStages")
    slots = (512 - accs * bn) // cols
    assert "constexpr int kSfAhead = kSfRing < kBsPairStages ? kSfRing : kBsPairStages;" in src
    return {"stages": stages, "ring": slots // kps, "ahead": min(slots // kps, stages)}


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "a phase received more arrivals than its count"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def completed(self, c):
        """A parity wait for completion number c (parity c & 1)."""
        assert self.phase <= c + 1, "a parity wait lapped its barrier"
        return self.phase == c + 1


def simulate(stages, ring, ahead, steps, seed):
    rnd = random.Random(seed)
    full = [Barrier(2 + 8) for _ in range(stages)]
    empty = [Barrier(1) for _ in range(stages)]
    prod, wr = [0, 0], [0] * 8
    issued, inflight, done = 0, [], -1
    slot_step = {}
    for _ in range(100000):
        if done == steps - 1:
            return
        acts = [("p", i) for i in range(2)
                if prod[i] < steps and (prod[i] < stages or empty[prod[i] % stages].completed(prod[i] // stages - 1))]
        acts += [("w", i) for i in range(8)
                 if wr[i] < steps and (wr[i] < ahead or empty[(wr[i] - ahead) % stages].completed((wr[i] - ahead) // stages))]
        if issued < steps and full[issued % stages].completed(issued // stages):
            acts.append(("m", 0))
        if inflight:
            acts.append(("c", 0))
        assert acts, "deadlock"
        kind, i = rnd.choice(acts)
        if kind == "p":
            full[prod[i] % stages].arrive()
            prod[i] += 1
        elif kind == "w":
            s = wr[i]
            prev = slot_step.get(s % ring)
            assert prev is None or prev == s or prev <= done, "scale slots rewritten before their MMAs completed"
            slot_step[s % ring] = s
            full[s % stages].arrive()
            wr[i] += 1
        elif kind == "m":
            assert slot_step.get(issued % ring) == issued, "MMAs would read another step's scales"
            inflight.append(issued)
            issued += 1
        else:
            done = inflight.pop(0)
            empty[done % stages].arrive()
    raise AssertionError("deadlock")


def test_kernel_protocol_under_random_schedules():
    k = kernel_constants()
    for seed in range(200):
        simulate(k["stages"], k["ring"], k["ahead"], 30, seed)


@pytest.mark.parametrize("ring", [2, 3, 4, 8])
def test_writer_bound_holds_for_every_slot_ring(ring):
    for seed in range(100):
        simulate(3, ring, min(ring, 3), 30, seed)


def test_writers_bounded_by_the_slot_ring_alone_break_the_operand_ring():
    """With more scale slots than operand stages, writers allowed as far ahead as the slot ring let
    their arrivals reach a `full` barrier whose previous phase is still open (what a version of the
    kernel did, and the GPU faulted)."""
    failures = 0
    for seed in range(100):
        try:
            simulate(3, 4, 4, 30, seed)
        except AssertionError:
            failures += 1
    assert failures > 50


# ------------------------------------------------------------------ scale ring

def ring_constants():
    src = open(GEMM).read()
    return {"slots": _const(src, "kScaleSlots"), "per_slot": _const(src, "kScaleGroupsPerSlot")}


def simulate_scale_ring(slots, per_slot, groups, tiles, seed, release_each_group=False):
    """The producer loads the scales of `per_slot` groups of one tile per ring slot, one slot ahead: the
    first at start-up, then one each time its operand loop enters a slot's first group; it waits for
    the slot's previous contents to have been consumed (`scale_empty`, parity of the refill).  Each of
    four writer warps waits for the slot (`scale_full`, parity) at a slot's first group, reads a group's
    words, and releases the slot after its last group of that tile.  Checks that every group's words
    come from the load of its own (tile, group), that no slot is refilled before all four writers
    released it, that no parity wait laps its barrier, and that nothing deadlocks."""
    rnd = random.Random(seed)
    pairs = -(-groups // per_slot)
    order = [(t, p) for t in range(tiles) for p in range(pairs)]  # slot loads in issue order
    full = [Barrier(1) for _ in range(slots)]
    empty = [Barrier(4) for _ in range(slots)]
    content = [None] * slots
    readers = [0] * slots  # writers yet to release the slot's current contents
    issued = 0
    prod_pos = 0            # the producer's position: groups entered so far (flattened)
    flat = [(t, g) for t in range(tiles) for g in range(groups)]
    wpos = [0] * 4          # each writer's next flattened group
    wcons = [0] * 4         # slots each writer has consumed

    def issue():
        nonlocal issued
        if issued >= len(order):
            return True
        s = issued % slots
        if issued >= slots and not empty[s].completed(issued // slots - 1):
            return False
        assert readers[s] == 0, "a slot was refilled before its writers released it"
        content[s] = order[issued]
        readers[s] = 4
        full[s].arrive()
        issued += 1
        return True

    assert issue()
    for _ in range(200000):
        if all(p == len(flat) for p in wpos) and prod_pos == len(flat):
            return
        acts = []
        if prod_pos < len(flat):
            acts.append(("p", 0))
        for w in range(4):
            if wpos[w] < len(flat):
                t, gr = flat[wpos[w]]
                s = wcons[w] % slots
                if gr % per_slot != 0 or full[s].completed(wcons[w] // slots):
                    acts.append(("w", w))
        assert acts, "deadlock"
        kind, i = rnd.choice(acts)
        if kind == "p":
            t, gr = flat[prod_pos]
            if gr % per_slot == 0:
                if not issue():
                    continue  # waiting for a slot to be released
            prod_pos += 1
        else:
            t, gr = flat[wpos[i]]
            s = wcons[i] % slots
            assert content[s] == (t, gr // per_slot), "a writer read another tile's or group's scales"
            wpos[i] += 1
            if release_each_group or gr % per_slot == per_slot - 1 or gr == groups - 1:
                readers[s] -= 1
                empty[s].arrive()
                wcons[i] += 1
    raise AssertionError("deadlock")


@pytest.mark.parametrize("groups", [1, 2, 3, 4, 5])
def test_scale_ring_under_random_schedules(groups):
    k = ring_constants()
    for seed in range(60):
        simulate_scale_ring(k["slots"], k["per_slot"], groups, 5, seed)


def test_scale_ring_releasing_each_group_breaks():
    """Writers that release a two-group slot after each group let the producer refill it (or the
    barrier run ahead) while its second group is still to be read."""
    failures = 0
    for seed in range(60):
        try:
            simulate_scale_ring(2, 2, 4, 5, seed, release_each_group=True)
        except AssertionError:
            failures += 1
    assert failures > 30
