"""A model of the deterministic dQ mode's turn protocol across CTAs, run under random schedules.

In the deterministic instance of the tensor-core backward (csrc/bwd_sm103.cu) every 128 x 128 dQ tile
of a query head receives the contributions of the key tiles that see it in key-tile order: the
tile has a turn counter (zeroed per call); the CTA of the t-th such key tile waits until the
counter equals t, issues its bulk reduce-adds, and one iteration later, once those adds are
complete, stores t + 1.  The kernel is free of deadlock by construction:
  * a CTA takes its logical index (which key tile of which group it owns) from a ticket counter
    in the workspace, in the order the CTAs actually start, whatever order the hardware
    dispatches the blocks in, and
  * a CTA only waits for CTAs of lower logical index (key tile outer in the logical index, and
    the key tiles of a query tile are consecutive from key_range's first one),
so every CTA waited for has started, and the lowest unfinished one never waits.

This model runs that protocol with a limited number of resident CTAs dispatched in a random
order, CTA pipelines that cannot stage the next dQ tile before their reduce warp released the
previous staging area, and adds that complete at random later times, and checks that no schedule
deadlocks and that every dQ tile receives its adds, completed, in key-tile order.  Planted
mistakes (passing a turn on before the adds complete, waiting for a higher index, taking the
logical index from the block index instead of the ticket) are caught.
"""
import random

import pytest


class TurnError(AssertionError):
    pass


def key_tiles_seeing(q, n_key_tiles, causal):
    """Key tiles whose keys some row of query tile q sees (S_q = S_k, 128-row tiles)."""
    return list(range(q + 1)) if causal else list(range(n_key_tiles))


def query_tiles_seen(kt, n_tiles, causal):
    return list(range(kt, n_tiles)) if causal else list(range(n_tiles))


class TurnModel:
    def __init__(self, groups, heads, n_tiles, causal, resident, rng, release_early=False,
                 wrong_order=False, ds_tiles=1, shuffle_dispatch=False, ticket=True):
        self.rng = rng
        self.shuffle_dispatch = shuffle_dispatch  # blocks dispatched in a random order
        self.ticket = ticket                      # logical index from the start-order ticket
        self.release_early = release_early
        self.ds_tiles = ds_tiles
        # block index = key tile * groups + group (key tile outer)
        self.ctas = []
        for kt in range(n_tiles):
            for grp in range(groups):
                its = []
                for q in reversed(query_tiles_seen(kt, n_tiles, causal)):  # last query tile first
                    for h in range(heads):
                        tiles = key_tiles_seeing(q, n_tiles, causal)
                        turn = tiles.index(kt)
                        if wrong_order:
                            turn = len(tiles) - 1 - turn
                        its.append(((grp, h, q), turn))
                self.ctas.append({"kt": kt, "its": its})
        self.counter = {}
        self.added = {}       # tile -> key tiles whose adds completed, in completion order
        self.expected = {}
        for grp in range(groups):
            for h in range(heads):
                for q in range(n_tiles):
                    self.expected[(grp, h, q)] = key_tiles_seeing(q, n_tiles, causal)
        self.resident = resident

    def cta_proc(self, c):
        """The reduce warp's loop of one CTA (the pipeline before it is folded into 'staged')."""
        cta = self.ctas[c]
        pending = []     # (tile, kt) adds issued, not yet complete
        prev = None      # turn to pass on: (tile, value)
        for i, (tile, turn) in enumerate(cta["its"]):
            yield ("staged",)                                  # dQ(i) staged by the drain
            yield ("wait_turn", tile, turn)
            handle = ("add", c, i)
            pending.append(handle)
            yield ("issue_add", handle, tile, cta["kt"])
            if self.release_early:                              # planted: no completion wait
                yield ("release", tile, turn + 1)
                continue
            if prev is not None:
                # the previous tile's adds are complete once at most this tile's are pending
                yield ("wait_complete", pending[:-1])
                yield ("release",) + prev
            pending = pending[-1:]
            prev = (tile, turn + 1)
        yield ("wait_complete", pending)
        if prev is not None and not self.release_early:
            yield ("release",) + prev

    def run(self):
        n = len(self.ctas)
        gens, blocked = {}, {}
        next_cta = 0  # blocks started so far (= the next ticket)
        order = list(range(n))  # physical block dispatched k-th
        if self.shuffle_dispatch:
            self.rng.shuffle(order)
        complete = set()
        inflight = []   # (handle, tile, kt) adds in flight
        steps = 0

        def start(c):
            gens[c] = self.cta_proc(c)
            blocked[c] = None
            step_cta(c)

        def ready(req):
            if req is None or req[0] == "staged":
                return True
            if req[0] == "wait_turn":
                return self.counter.get(req[1], 0) == req[2]
            if req[0] == "wait_complete":
                return all(h in complete for h in req[1])
            raise AssertionError(req)

        def step_cta(c):
            while True:
                try:
                    req = next(gens[c])
                except StopIteration:
                    del gens[c]
                    return
                if req[0] == "issue_add":
                    inflight.append(req[1:])
                    continue
                if req[0] == "release":
                    self.counter[req[1]] = req[2]
                    continue
                blocked[c] = req
                if req[0] == "staged":
                    return  # time passes
                if ready(req):
                    continue
                return

        while next_cta < n or gens or inflight:
            steps += 1
            if steps > 200000:
                raise TurnError("no progress")
            while next_cta < n and len(gens) < self.resident:
                # with the ticket the k-th started block owns logical CTA k; without it, the
                # block owns the logical CTA of its own block index
                start(next_cta if self.ticket else order[next_cta])
                next_cta += 1
            choices = [("cta", c) for c in gens if ready(blocked[c])]
            choices += [("add", k) for k in range(len(inflight))]
            if not choices:
                raise TurnError("deadlock: " + ", ".join(f"CTA {c} at {blocked[c]}" for c in gens))
            kind, key = self.rng.choice(choices)
            if kind == "cta":
                blocked[key] = None
                step_cta(key)
            else:
                handle, tile, kt = inflight.pop(key)
                complete.add(handle)
                self.added.setdefault(tile, []).append(kt)
        for tile, kts in self.expected.items():
            if self.added.get(tile, []) != kts:
                raise TurnError(f"tile {tile} got adds {self.added.get(tile)} instead of {kts}")
        return True


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("resident", [1, 3, 8])
def test_turns_add_in_key_tile_order_without_deadlock(causal, resident):
    rng = random.Random(31 + resident + 7 * causal)
    for _ in range(150):
        TurnModel(groups=2, heads=2, n_tiles=rng.choice([1, 2, 3, 4]), causal=causal,
                  resident=resident, rng=random.Random(rng.random()), shuffle_dispatch=True).run()


def test_model_catches_block_index_order_under_out_of_order_dispatch():
    # without the ticket, a block dispatched early may own a late logical index and wait for a
    # block that cannot become resident: caught as a deadlock on some schedule
    rng = random.Random(5)
    caught = 0
    for _ in range(100):
        try:
            TurnModel(1, 1, 4, False, 2, random.Random(rng.random()), shuffle_dispatch=True,
                      ticket=False).run()
        except TurnError:
            caught += 1
    assert caught > 0


def test_model_catches_a_turn_passed_before_the_adds_complete():
    rng = random.Random(3)
    caught = 0
    for _ in range(200):
        try:
            TurnModel(2, 2, 4, False, 8, random.Random(rng.random()), release_early=True).run()
        except TurnError:
            caught += 1
    assert caught > 0


def test_model_catches_waiting_for_a_higher_block_index():
    # turns handed out in descending key-tile order: a CTA waits for a later-dispatched one,
    # which deadlocks as soon as fewer CTAs are resident than the chain needs
    rng = random.Random(4)
    caught = 0
    for _ in range(50):
        try:
            TurnModel(1, 1, 4, False, 2, random.Random(rng.random()), wrong_order=True).run()
        except TurnError:
            caught += 1
    assert caught == 50
