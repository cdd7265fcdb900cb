"""Model of the decode kernel's tile ring (CPU only).

The kernel streams tile t into stage t % STAGES; consumer warp t % W reads
it after a parity wait on the stage's "full" barrier and releases it on the
"empty" barrier; the producer refills a stage after a parity wait on "empty".
A parity wait succeeds when the most recently completed phase has the asked
parity, so it cannot tell phase u from phase u + 2. This model replays random
interleavings with those semantics and checks that every consumer reads the
tile it waited for. Stage counts that are a multiple of the warp count (each
stage owned by one warp) are safe; others are not, which is why the kernel
asserts STAGES % W == 0 at compile time.
"""
import random

import pytest


def replay(stages, warps, ntiles, seed):
    rnd = random.Random(seed)
    full = [0] * stages           # completed phases per barrier
    empty = [0] * stages
    in_flight = {}
    content = [None] * stages
    issued = 0
    nxt = list(range(warps))

    def done(completed, parity):
        return completed > 0 and ((completed - 1) & 1) == parity

    wrong = 0
    for _ in range(100_000):
        acts = []
        if issued < ntiles:
            t = issued
            if t < stages or done(empty[t % stages], (t // stages - 1) & 1):
                acts.append(("issue", t))
        acts += [("land", s) for s in in_flight]
        acts += [("take", w) for w in range(warps)
                 if nxt[w] < ntiles and done(full[nxt[w] % stages], (nxt[w] // stages) & 1)]
        if not acts:
            break
        kind, x = rnd.choice(acts)
        if kind == "issue":
            if x % stages in in_flight:
                wrong += 1
            in_flight[x % stages] = x
            issued += 1
        elif kind == "land":
            content[x] = in_flight.pop(x)
            full[x] += 1
        else:
            t = nxt[x]
            wrong += content[t % stages] != t
            empty[t % stages] += 1
            nxt[x] += warps
    finished = all(n >= ntiles for n in nxt)
    return wrong, finished


@pytest.mark.parametrize("stages,warps", [(4, 4), (8, 4), (12, 4), (4, 2), (6, 2), (3, 1)])
def test_owned_stages_are_safe(stages, warps):
    for seed in range(200):
        wrong, finished = replay(stages, warps, 40, seed)
        assert wrong == 0 and finished, seed


def test_shared_stages_break():
    bad = sum(replay(6, 4, 40, seed)[0] > 0 for seed in range(200))
    assert bad > 0
