"""A CPU model of the tensor-core GEMM's barrier protocol (gemm_tc.cu).

The roles, replayed in the kernel's order under random schedules and random completion
times of the asynchronous operations (TMA copies, tcgen05.commit arrivals):

  * the producer walks the CTA's tiles and their K steps (`it` counts them all) and loads
    step `it` into ring stage it % S once that stage's previous fill has been released
    (empty), completing full asynchronously;
  * the MMA issuer takes tile tc into accumulator tc % 2 after the epilogue released that
    accumulator's previous tile (acc_empty), waits every step's full, releases each stage
    by a commit (arriving when its MMAs complete) and commits acc_full after the tile;
  * four epilogue warps wait acc_full of each tile's accumulator and arrive on its
    acc_empty (the kernel counts the 128 threads; the model counts the four warps).

Commits from the issuing thread arrive in issue order.  The model checks that nothing
deadlocks and that every wait starts while its barrier is at most one phase from the
awaited one (a waiter two phases behind would take a later phase for its own).
"""
import random

import pytest

EPI_WARPS = 4


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


def run_protocol(n_tiles, k_steps, stages, rng, mistake=None, lazy=False):
    B = {}
    for s in range(stages):
        B[f"full{s}"] = Barrier(f"full{s}", 1)
        B[f"empty{s}"] = Barrier(f"empty{s}", 1)
    for b in range(2):
        B[f"acc_full{b}"] = Barrier(f"acc_full{b}", 1)
        B[f"acc_empty{b}"] = Barrier(f"acc_empty{b}", 1 if mistake == "acc_empty_count_one"
                                     else EPI_WARPS)

    def acc(tc):
        return 0 if mistake == "one_accumulator" else tc % 2

    def producer():
        it = 0
        for _ in range(n_tiles):
            for _ in range(k_steps):
                s = it % stages
                if it >= stages:
                    yield ("wait", f"empty{s}", it // stages - 1)
                yield ("async", [f"full{s}"])
                it += 1

    def issuer():
        it = 0
        for tc in range(n_tiles):
            if tc >= 2 and mistake != "skip_acc_empty_wait":
                yield ("wait", f"acc_empty{acc(tc)}", tc // 2 - 1)
            for _ in range(k_steps):
                s = it % stages
                yield ("wait", f"full{s}", it // stages)
                yield ("async", [f"empty{s}"])
                it += 1
            yield ("async", [f"acc_full{acc(tc)}"])

    def epilogue():
        for tc in range(n_tiles):
            yield ("wait", f"acc_full{acc(tc)}", tc // 2)
            yield ("arrive", f"acc_empty{acc(tc)}")

    actors = [producer(), issuer()] + [epilogue() for _ in range(EPI_WARPS)]
    streams = [[] for _ in actors]
    current = [next(a, None) for a in actors]
    slow = 2 + rng.randrange(EPI_WARPS)            # a rarely scheduled epilogue warp

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
                raise Deadlock(f"tiles={n_tiles} k_steps={k_steps} stages={stages}: "
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
def test_gemm_protocol_never_deadlocks_or_aliases(seed):
    rng = random.Random(seed)
    for _ in range(8):
        run_protocol(n_tiles=rng.randint(1, 9), k_steps=rng.randint(1, 9),
                     stages=rng.randint(2, 4), rng=rng, lazy=seed % 2 == 1)


@pytest.mark.parametrize("mistake", ["skip_acc_empty_wait", "one_accumulator",
                                     "acc_empty_count_one"])
def test_model_catches_planted_mistakes(mistake):
    """Plausible mistakes must fail the model: the issuer overwriting an accumulator the
    epilogue has not drained; both tiles of a pair sent to one accumulator while the
    waits still count two; an acc_empty barrier initialised for one arrival while every
    epilogue warp arrives."""
    rng = random.Random(5)
    with pytest.raises((AssertionError, Deadlock)):
        for k in range(40):
            run_protocol(n_tiles=8, k_steps=3, stages=4, rng=rng, mistake=mistake,
                         lazy=k % 2 == 1)
