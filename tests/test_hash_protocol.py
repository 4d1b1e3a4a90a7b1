"""A CPU model of the tensor-core hash kernel's barrier protocol.

The roles, replayed in the kernel's order under random schedules and random completion
times of the asynchronous operations (TMA copies, tcgen05.commit arrivals):

  * the producer loads token tile `it` into stage it % X after that stage's previous
    tile is released (x_empty), completing x_full asynchronously;
  * MMA issuer e (one per epilogue warpgroup) waits for every tile's stage; for its own
    tiles (it % 2 == e) it runs the tile's chunks through the warpgroup's accumulators
    2e and 2e + 1 in turn (use u of the warpgroup goes to 2e + u % 2), each after the
    epilogue released that accumulator's previous chunk (tm_empty), committing tm_full;
    it releases the stage by a commit after its chunks (own tile) or a plain arrival;
  * the norm warp (first group only) reads every stage and arrives on x_empty;
  * epilogue warpgroup e (four warps) takes the tiles it % 2 == e: per chunk each of its
    warps waits tm_full of the chunk's accumulator and arrives on its tm_empty (the
    kernel counts the warpgroup's 128 threads; the model counts its four warps).

Commits from one thread arrive in issue order.  The model checks that nothing deadlocks
and that every wait starts while its barrier is at most one phase from the awaited one.
"""
import random

import pytest

GROUPS = 2        # epilogue warpgroups = MMA issuers
ACCS = 2          # accumulators per warpgroup
GROUP_WARPS = 4


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


def run_protocol(n_tiles, nch, stages, with_norm, rng, mistake=None, lazy=False):
    B = {"r_full": Barrier("r_full", 1)}
    for s in range(stages):
        B[f"x_full{s}"] = Barrier(f"x_full{s}", 1)
        counted = with_norm and mistake != "norm_not_counted"
        B[f"x_empty{s}"] = Barrier(f"x_empty{s}", GROUPS + (1 if counted else 0))
    for b in range(GROUPS * ACCS):
        B[f"tm_full{b}"] = Barrier(f"tm_full{b}", 1)
        B[f"tm_empty{b}"] = Barrier(f"tm_empty{b}", GROUP_WARPS)

    def acc(e, use):
        return ACCS * e + (0 if mistake == "one_accumulator" else use % ACCS)

    def producer():
        yield ("async", ["r_full"])
        for it in range(n_tiles):
            s = it % stages
            if it >= stages:
                yield ("wait", f"x_empty{s}", it // stages - 1)
            yield ("async", [f"x_full{s}"])

    def issuer(e):
        yield ("wait", "r_full", 0)
        for it in range(n_tiles):
            s = it % stages
            yield ("wait", f"x_full{s}", it // stages)
            if it % GROUPS == e:
                for k in range(nch):
                    use = (it // GROUPS) * nch + k
                    if use >= ACCS and mistake != "skip_tm_empty_wait":
                        yield ("wait", f"tm_empty{acc(e, use)}", use // ACCS - 1)
                    yield ("async", [f"tm_full{acc(e, use)}"])
                yield ("async", [f"x_empty{s}"])
            else:
                yield ("arrive", f"x_empty{s}")

    def norm():
        for it in range(n_tiles):
            s = it % stages
            yield ("wait", f"x_full{s}", it // stages)
            yield ("arrive", f"x_empty{s}")

    def epilogue(e):
        for it in range(n_tiles):
            if it % GROUPS != e:
                continue
            for k in range(nch):
                use = (it // GROUPS) * nch + k
                yield ("wait", f"tm_full{acc(e, use)}", use // ACCS)
                yield ("arrive", f"tm_empty{acc(e, use)}")

    actors = [producer()] + [issuer(e) for e in range(GROUPS)]
    n_fixed = len(actors)
    actors += [epilogue(e) for e in range(GROUPS) for _ in range(GROUP_WARPS)]
    if with_norm:
        actors.append(norm())
    streams = [[] for _ in actors]
    current = [next(a, None) for a in actors]
    slow = n_fixed + rng.randrange(GROUPS * GROUP_WARPS)   # a rarely scheduled epilogue warp

    def blocked(op):
        if op is None or op[0] != "wait":
            return False
        bar = B[op[1]]
        assert op[2] <= bar.phases <= op[2] + 1, (
            f"{op[1]}: waiter for phase {op[2]} while {bar.phases} phases completed")
        return bar.phases <= op[2]

    for _ in range(500000):
        runnable = [i for i, op in enumerate(current) if op is not None and not blocked(op)]
        pending = [i for i, st in enumerate(streams) if st]
        if not runnable and not pending:
            if any(op is not None for op in current):
                raise Deadlock(f"tiles={n_tiles} nch={nch} stages={stages}: "
                               f"stuck at {[op for op in current if op is not None]}")
            return
        if pending and (not runnable or rng.random() < 0.3):
            i = rng.choice(pending)
            for name in streams[i].pop(0):
                B[name].arrive()
            continue
        if lazy:
            i = rng.choices(runnable, weights=[0.02 if k == slow else 1.0 for k in runnable])[0]
        else:
            i = rng.choice(runnable)
        op = current[i]
        if op[0] == "arrive":
            B[op[1]].arrive()
        elif op[0] == "async":
            streams[i].append(op[1])
        current[i] = next(actors[i], None)
    raise AssertionError("model did not finish")


@pytest.mark.parametrize("seed", range(30))
def test_hash_protocol_never_deadlocks_or_aliases(seed):
    rng = random.Random(seed)
    for _ in range(8):
        run_protocol(n_tiles=rng.randint(1, 23), nch=rng.randint(1, 5), stages=rng.randint(2, 4),
                     with_norm=rng.random() < 0.5, rng=rng, lazy=seed % 2 == 1)


@pytest.mark.parametrize("mistake", ["norm_not_counted", "skip_tm_empty_wait", "one_accumulator"])
def test_model_catches_planted_mistakes(mistake):
    """Plausible mistakes must fail the model: a stage's release count that leaves out the
    norm warp (the producer may refill a stage the norm warp still reads); an MMA issuer
    overwriting an accumulator without waiting for the epilogue to release it; or both
    uses of a warpgroup sent to one accumulator while the waits still count two."""
    rng = random.Random(3)
    with pytest.raises((AssertionError, Deadlock)):
        for k in range(40):
            run_protocol(n_tiles=16, nch=4, stages=3, with_norm=True, rng=rng, mistake=mistake,
                         lazy=k % 2 == 1)
