"""A CPU model of the tensor-core attention kernel's barrier protocol.

The attention kernel coordinates its warps through mbarriers only.  This model replays
each role's barrier operations in the kernel's order for random work splits, under random
schedules and random completion times of the asynchronous operations:

  * a slot's metadata warp and its copy warps each wait for the slot's release (empty),
    then arrive on `full` (the copy warps asynchronously, once their copies land);
  * the S issuer needs the tile's chunks, waits for its S buffer to be free (pv_done of
    the tile two back) and commits s_full;
  * the P V issuer needs the chunks, waits for P (p_full) and for the epilogue to free
    O (o_empty), then commits o_full, pv_done and the release of the chunks whose last
    use this was;
  * each softmax warp needs the chunks, waits for S, arrives on p_full, then runs the
    epilogue of the previous tile (waits o_full and p_full, arrives on o_empty).

A commit (tcgen05.commit, cp.async.mbarrier.arrive) arrives when everything its thread
issued before it has completed, so each asynchronous stream completes in order.  An
mbarrier wait on parity p passes while the number of completed phases has the other
parity (PTX semantics).  The model checks that no schedule deadlocks and that every
wait starts while the barrier is at most one phase from the awaited one: neither two
phases behind (the parity would then name a later phase: the hazard that broke an
earlier version of the kernel) nor still finishing the phase before the awaited one
(the parity of that earlier, completed phase would then pass the wait at once).
"""
import random

import pytest

SLOTS = 6           # chunk ring
COPY_WARPS = 9      # row copiers (plus one metadata warp)
SOFTMAX = 2         # softmax warps modelled (the kernel has 16; all run the same program)


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phases = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than its count"
        if self.pending == 0:
            self.phases += 1
            self.pending = self.count


class Deadlock(Exception):
    pass


def items_of(nch, n_seg, u0, u1):
    """The CTA's (seg, tb, te) items for units [u0, u1), as the kernel walks them."""
    tps = (nch + 1) // 2
    out, u = [], u0
    while u < u1:
        seg = u // tps
        tb = u - seg * tps
        te = min(tb + (u1 - u), tps)
        out.append((seg, tb, te))
        u += te - tb
    return out


def chunks(nch, tb, te):
    return range(2 * tb - 1 if tb > 0 else 0, min(2 * te, nch))


def tile_chunks(nch, t, tb):
    cs = ([2 * t - 1] if (t == tb and tb > 0) else []) + [2 * t]
    if 2 * t + 1 < nch:
        cs.append(2 * t + 1)
    return cs


def run_protocol(nch, items, rng, slots=SLOTS, mistake=None, lazy_softmax=False):
    """lazy_softmax: schedule the softmax warps rarely (the other roles race ahead)."""
    SLOTS = slots  # noqa: N806 (the ring size of this run)
    B = {}
    for s in range(SLOTS):
        B[f"full{s}"] = Barrier(f"full{s}", 1 + COPY_WARPS)
        B[f"empty{s}"] = Barrier(f"empty{s}", 1)
    for b in range(2):
        B[f"s_full{b}"] = Barrier(f"s_full{b}", 1)
        B[f"p_full{b}"] = Barrier(f"p_full{b}", SOFTMAX)
        B[f"pv_done{b}"] = Barrier(f"pv_done{b}", 1)
    B["o_full"] = Barrier("o_full", 1)
    B["o_empty"] = Barrier("o_empty", SOFTMAX)

    # Ops: ("wait", barrier, absolute phase) -- passes once that phase has completed;
    # ("arrive", barrier); ("async", [barriers]) -- arrives later, in stream order.
    def loader(is_meta):
        fills = [0] * SLOTS
        for seg, tb, te in items:
            for c in chunks(nch, tb, te):
                s = c % SLOTS
                if fills[s] > 0:
                    yield ("wait", f"empty{s}", fills[s] - 1)
                fills[s] += 1
                yield ("arrive", f"full{s}") if is_meta else ("async", [f"full{s}"])

    def need(fills, c):
        s = c % SLOTS
        op = ("wait", f"full{s}", fills[s])
        fills[s] += 1
        return op

    def s_issuer():
        fills, ctr = [0] * SLOTS, 0
        for seg, tb, te in items:
            for t in range(tb, te):
                for c in tile_chunks(nch, t, tb):
                    yield need(fills, c)
                b = ctr & 1
                if ctr >= 2:
                    yield ("wait", f"pv_done{b}", (ctr - 2) >> 1)
                yield ("async", [f"s_full{b}"])
                ctr += 1

    def pv_issuer():
        fills, q = [0] * SLOTS, 0
        for seg, tb, te in items:
            for t in range(tb, te):
                for c in tile_chunks(nch, t, tb):
                    yield need(fills, c)
                b = q & 1
                yield ("wait", f"p_full{b}", q >> 1)
                if q >= 1:
                    yield ("wait", "o_empty", q - 1)
                rel = ([f"empty{(2 * t - 1) % SLOTS}"] if t > 0 else []) + [f"empty{(2 * t) % SLOTS}"]
                if (t == te - 1 or mistake == "release_odd_chunk_early") and 2 * t + 1 < nch:
                    rel.append(f"empty{(2 * t + 1) % SLOTS}")
                yield ("async", ["o_full", f"pv_done{b}"] + rel)
                q += 1

    def softmax():
        fills, ctr = [0] * SLOTS, 0

        def epilogue(q):
            yield ("wait", "o_full", q)
            yield ("wait", f"p_full{q & 1}", q >> 1)
            yield ("arrive", "o_empty")

        for seg, tb, te in items:
            for t in range(tb, te):
                for c in tile_chunks(nch, t, tb):
                    yield need(fills, c)
                b = ctr & 1
                yield ("wait", f"s_full{b}", ctr >> 1)
                yield ("arrive", f"p_full{b}")
                if ctr >= 1:
                    yield from epilogue(ctr - 1)
                ctr += 1
        if ctr >= 1:
            yield from epilogue(ctr - 1)

    actors = [loader(True)] + [loader(False) for _ in range(COPY_WARPS)]
    actors += [s_issuer(), pv_issuer()]
    n_fixed = len(actors)               # the actors before this index are not softmax warps
    actors += [softmax() for _ in range(SOFTMAX)]
    streams = [[] for _ in actors]      # pending asynchronous arrival groups, in order
    current = [next(a, None) for a in actors]

    def blocked(op):
        if op is None or op[0] != "wait":
            return False
        bar = B[op[1]]
        assert op[2] <= bar.phases <= op[2] + 1, (
            f"{op[1]}: waiter for phase {op[2]} while {bar.phases} phases completed")
        return bar.phases <= op[2]

    steps = 0
    while True:
        steps += 1
        assert steps < 200000
        runnable = [i for i, op in enumerate(current) if op is not None and not blocked(op)]
        pending = [i for i, st in enumerate(streams) if st]
        if not runnable and not pending:
            if any(op is not None for op in current):
                stuck = [op for op in current if op is not None]
                raise Deadlock(f"nch={nch} items={items}: stuck at {stuck}")
            return
        # complete an asynchronous group now and then (in its stream's order)
        if pending and (not runnable or rng.random() < 0.3):
            i = rng.choice(pending)
            for name in streams[i].pop(0):
                B[name].arrive()
            continue
        if lazy_softmax:
            i = rng.choices(runnable, weights=[0.02 if k >= n_fixed else 1.0 for k in runnable])[0]
        else:
            i = rng.choice(runnable)
        op = current[i]
        if op[0] == "arrive":
            B[op[1]].arrive()
        elif op[0] == "async":
            streams[i].append(op[1])
        current[i] = next(actors[i], None)


@pytest.mark.parametrize("seed", range(40))
def test_attention_protocol_never_deadlocks_or_aliases(seed):
    rng = random.Random(seed)
    for _ in range(10):
        nch = rng.randint(1, 11)
        tps = (nch + 1) // 2
        n_seg = rng.randint(1, 3)
        total = n_seg * tps
        u0 = rng.randrange(total)
        u1 = rng.randint(u0 + 1, total)
        run_protocol(nch, items_of(nch, n_seg, u0, u1), rng, lazy_softmax=seed % 2 == 1)


@pytest.mark.parametrize("mistake,slots", [("release_odd_chunk_early", SLOTS), (None, 2)])
def test_model_catches_planted_mistakes(mistake, slots):
    """Plausible mistakes must fail the model: the P V issuer also releasing a tile's odd
    chunk, which the next tile still reads as its look-back (the slot gets released
    twice and refilled while in use); or a ring too small for the three-chunk window."""
    rng = random.Random(1)
    with pytest.raises((AssertionError, Deadlock)):
        for _ in range(50):
            run_protocol(9, items_of(9, 2, 0, 10), rng, slots=slots, mistake=mistake)
