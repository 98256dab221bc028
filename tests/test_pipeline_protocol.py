"""A host model of the score kernel's streaming pipeline protocol (index_topk.cu: the
scheduler warp, the two producer warps, the MMA warp and the two epilogue groups), with
the mbarrier parity rule: a wait for parity p returns once the barrier's phase with
parity p has completed, so a waiter must never fall two phases behind its barrier.

The model keeps the kernel's ring sizes and its phase arithmetic (8 tile records, 4
stages per producer, 8 accumulators whose MMA commit also frees the stage, 16 scale
slots, 2 query-image buffers, one end record per producer) and runs the roles with
random speeds, random request runs and random pauses at the epilogue's request
switches (its histogram flush).  It checks that every role finishes; a variant that
commits the MMAs once per pair of tiles shows the model finds a missed phase when the
pair's second tile is the end marker and its commit skips the accumulator wait."""

import random

import pytest


class _Bar:
    """An mbarrier with an arrival count and a phase counter."""

    def __init__(self, count=1):
        self.count = self.pending = count
        self.phase = 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


def _run(tiles, seed, paired=False, end_wait=True, slow=None, switch_pause=None):
    """Runs the roles over one block's tile sequence (request id per tile); returns
    "ok" or a description of the roles left waiting."""
    rnd = random.Random(seed)
    K_STAGES, K_ACCS, K_REC, K_SS = 4, 8, 8, 16
    full = [[_Bar() for _ in range(K_STAGES)] for _ in range(2)]
    accfull = [_Bar() for _ in range(K_ACCS)]
    accempty = [_Bar() for _ in range(K_ACCS)]
    qfull, qempty = [_Bar(), _Bar()], [_Bar(), _Bar()]
    sfull = [_Bar() for _ in range(K_SS)]
    sempty = [_Bar() for _ in range(K_SS)]
    rfull = [_Bar() for _ in range(K_REC)]
    rempty = [_Bar() for _ in range(K_REC)]
    rec, tinfo = [None] * K_REC, [None] * K_SS

    def tile_done(i):   # the barrier that completes once tile i's MMAs have
        return accfull[(i >> 1) % (K_ACCS // 2)] if paired else accfull[i % K_ACCS]

    now = [0]
    events = []          # asynchronous completions: (time, action)
    pending_mma = set()
    commits = []         # (barrier, MMAs it tracks)
    serial = [0]

    def later(fn):
        events.append((now[0] + rnd.randint(1, 30), fn))

    def settle():
        for c in list(commits):
            if not (c[1] & pending_mma):
                commits.remove(c)
                c[0].arrive()

    def mma_issue():
        serial[0] += 1
        k = serial[0]
        pending_mma.add(k)

        def fin():
            pending_mma.discard(k)
            settle()
        later(fin)

    def mma_commit(bar):
        commits.append((bar, set(pending_mma)))
        settle()

    def scheduler():
        nreq, cur, i = 0, None, 0
        for t in list(tiles) + [-1, -1]:
            if t >= 0 and t != cur:   # a new request's query image into buffer nreq % 2
                b = nreq & 1
                if nreq >= 2:
                    yield lambda b=b, ph=((nreq >> 1) - 1) & 1: qempty[b].done(ph)
                later(qfull[b].arrive)
                nreq += 1
                cur = t
            rs, u = i % K_REC, i // K_REC
            if u > 0:
                yield lambda rs=rs, ph=(u - 1) & 1: rempty[rs].done(ph)
            rec[rs] = t
            rfull[rs].arrive()
            i += 1

    def producer(pw):
        posts, i = 0, pw
        while True:
            rs = i % K_REC
            yield lambda rs=rs, ph=(i // K_REC) & 1: rfull[rs].done(ph)
            t = rec[rs]
            rempty[rs].arrive()
            s, rnd_ = posts % K_STAGES, posts // K_STAGES
            if rnd_ > 0:   # the stage is free once the tile that used it has had its MMAs
                yield lambda i=i, ph=(rnd_ - 1) & 1: tile_done(i).done(ph)
            ss, su = i % K_SS, i // K_SS
            if su > 0:
                yield lambda ss=ss, ph=(su - 1) & 1: sempty[ss].done(ph)
            tinfo[ss] = t
            later(full[pw][s].arrive)
            later(sfull[ss].arrive)
            posts += 1
            if t < 0:
                return
            i += 2

    def mma():
        nreq, qb, cur, i = 0, 0, None, 0
        while True:
            pw, ip = i & 1, i >> 1
            s = ip % K_STAGES
            yield lambda pw=pw, s=s, ph=(ip // K_STAGES) & 1: full[pw][s].done(ph)
            t = tinfo[i % K_SS]
            if t < 0:
                if paired and (i & 1):   # the pair's first tile alone
                    c, use = i % K_ACCS, i // K_ACCS
                    if end_wait and use > 0:
                        yield lambda c=c, ph=(use - 1) & 1: accempty[c].done(ph)
                    mma_commit(tile_done(i))
                return
            if t != cur:
                if cur is not None:
                    mma_commit(qempty[qb])
                qb = nreq & 1
                yield lambda qb=qb, ph=(nreq >> 1) & 1: qfull[qb].done(ph)
                nreq += 1
                cur = t
            c, use = i % K_ACCS, i // K_ACCS
            if use > 0:
                yield lambda c=c, ph=(use - 1) & 1: accempty[c].done(ph)
            for _ in range(4):
                mma_issue()
            if not paired or (i & 1):
                mma_commit(tile_done(i))
            i += 1

    def epilogue(g):
        i, cur = g, None
        while True:
            ss = i % K_SS
            yield lambda ss=ss, ph=(i // K_SS) & 1: sfull[ss].done(ph)
            t = tinfo[ss]
            sempty[ss].arrive()
            if t < 0:
                return
            if t != cur:   # request switch: the flush, during which no barrier is looked at
                cur = t
                pause = switch_pause(g, t) if switch_pause else rnd.choice([0, 5, 50, 400, 3000])
                until = now[0] + pause
                wake = (lambda u=until: now[0] >= u)
                wake.timer = True
                yield wake
            yield lambda i=i, ph=(i // K_ACCS) & 1: tile_done(i).done(ph)
            accempty[i % K_ACCS].arrive()
            i += 2

    roles = {"scheduler": scheduler(), "producer0": producer(0), "producer1": producer(1), "mma": mma(),
             "epilogue0": epilogue(0), "epilogue1": epilogue(1)}
    speed = {k: rnd.choice([1.0, 1.0, 0.5, 0.1]) for k in roles}
    if slow:
        speed.update(slow)
    waits = {k: None for k in roles}
    alive = set(roles)
    for _ in range(400_000):
        progressed = False
        for k in rnd.sample(sorted(alive), len(alive)):
            if rnd.random() > speed[k]:
                continue
            while True:
                w = waits[k]
                if w is not None and not w():
                    break
                try:
                    waits[k] = next(roles[k])
                    progressed = True
                except StopIteration:
                    alive.discard(k)
                    progressed = True
                    break
        if not alive:
            return "ok"
        now[0] += 1
        ready = any(waits[k] is None or waits[k]() for k in alive)
        timer = any(getattr(waits[k], "timer", False) for k in alive)
        if progressed or ready:
            if events and rnd.random() < 0.5:
                events.sort(key=lambda e: e[0])
                t, fn = events.pop(0)
                now[0] = max(now[0], t)
                fn()
            continue
        if events:
            events.sort(key=lambda e: e[0])
            t, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
        elif not timer:
            return "waiting: " + ", ".join(sorted(alive))
    return "too long"


def _tiles(rnd):
    """One block's tile sequence: runs of tiles of successive requests (chunks of up to
    four, requests switching often), as the scheduler hands them out."""
    n = rnd.randint(1, 48)
    out, r = [], 0
    while len(out) < n:
        out += [r] * rnd.choice([1, 1, 2, 3, 4, 5, 8, 13])
        r += 1
    return out[:n]


def test_stream_protocol_completes_under_random_schedules():
    rnd = random.Random(2026)
    for case in range(120):
        tiles = _tiles(rnd)
        res = _run(tiles, seed=case)
        assert res == "ok", (case, tiles, res)


@pytest.mark.parametrize("end_wait,expect", [(False, "waiting"), (True, "ok")])
def test_model_finds_the_paired_commit_hazard(end_wait, expect):
    """One MMA commit per pair of tiles: with the end marker second in a pair and a
    commit that does not wait for the slot's accumulator, the barrier can run two phases
    ahead of an epilogue group paused at a request switch, which then waits for ever."""
    tiles = [2, 2, 2, 3, 3, 3, 3, 3, 3, 3, 3]
    hits = 0
    for seed in range(40):
        res = _run(tiles, seed, paired=True, end_wait=end_wait,
                   slow={k: 1.0 for k in ("scheduler", "producer0", "producer1", "mma", "epilogue0", "epilogue1")},
                   switch_pause=lambda g, t: 20000 if (g == 1 and t == 3) else 0)
        hits += res.startswith(expect)
    assert hits == 40 if expect == "ok" else hits > 0
