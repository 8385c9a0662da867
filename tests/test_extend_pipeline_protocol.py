"""Model check of the extend-attention kernel's synchronisation protocol (host only).

The kernel (csrc/extend_attention.cu) runs on a pair of CTAs (ranks 0 and 1 of
a cluster) around mbarriers.  In each CTA, loader warps fill that CTA's half of
a K/V ring and write its Q; softmax warps read its S rows, rescale its O and
write its P.  One thread of rank 0 issues the pair's tensor-core MMAs (S = Q K^T
into two S buffers, O += P V), which read both CTAs' halves and write both
CTAs' S and O, and commits each group to the mbarrier of that name in both
CTAs (multicast).  The loaders and softmax warps of both CTAs arrive on rank
0's barriers (q_full, kv_full, p_full take one arrival per CTA here).  The
tensor core finishes issued MMAs in order, asynchronously.  This model replays
each role's sequence of waits, arrivals, commits and buffer accesses, in the
kernel's order, under random interleavings, and checks:

- every wait targets the completion it means: the barrier has at most one
  more completed phase than the one waited for (else the parity would alias);
- no buffer is overwritten while an earlier user may still read it (K/V
  stages, S buffers, P, O), and every read sees the tile it expects;
- every interleaving finishes (no deadlock).
"""
import random

import pytest

STAGES, SBUF = 6, 2
RANKS = (0, 1)


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0  # done = completed phases

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


def both(name):
    return [f"{name}@{r}" for r in RANKS]


def roles(n):
    """The kernel's roles as action lists (see the module docstring); a
    buffer or barrier name ends in @rank, the CTA that holds it."""
    progs = {}
    for r in RANKS:
        loader = [("write", f"Q@{r}", 0), ("arrive", "q_full@0")]
        for i in range(n):
            s = i % STAGES
            if i >= STAGES:
                loader.append(("wait", f"kv_empty{s}@{r}", i // STAGES - 1))
            loader += [("write", f"KV{s}@{r}", i), ("arrive", f"kv_full{s}@0")]
        softmax = []
        for i in range(n):
            softmax += [("wait", f"s_full{i % SBUF}@{r}", i // SBUF), ("read", f"S{i % SBUF}@{r}", i)]
            if i >= 1:
                softmax += [("wait", f"o_done@{r}", i - 1), ("write", f"O@{r}", i)]   # the lazy rescale of O
            softmax += [("write", f"P@{r}", i), ("arrive", "p_full@0")]
        softmax += [("wait", f"o_done@{r}", n - 1), ("read", f"O@{r}", n)]
        progs[f"loader{r}"], progs[f"softmax{r}"] = loader, softmax
    mma = [("wait", "q_full@0", 0)]
    for i in range(n + 1):
        if i < n:
            s = i % STAGES
            mma += [("wait", f"kv_full{s}@0", i // STAGES),
                    ("issue", "S", i, [(b, 0) for b in both("Q")] + [(b, i) for b in both(f"KV{s}")],
                     [(b, i) for b in both(f"S{i % SBUF}")]),
                    ("commit", both(f"s_full{i % SBUF}"))]
        if i >= 1:
            pi = i - 1
            mma += [("wait", "p_full@0", pi),
                    ("issue", "PV", pi, [(b, pi) for b in both("P")] + [(b, pi) for b in both(f"KV{pi % STAGES}")],
                     [(b, pi) for b in both("O")]),
                    ("commit", both("o_done"))]
            if pi + STAGES < n:
                mma.append(("commit", both(f"kv_empty{pi % STAGES}")))
    mma += [("commit", ["drain@0"]), ("wait", "drain@0", 0)]
    progs["mma"] = mma
    return progs


def run(n, seed):
    rng = random.Random(seed)
    # rank 0's q_full, kv_full and p_full take one arrival per CTA
    bars = {"q_full@0": Barrier(2), "p_full@0": Barrier(2), "drain@0": Barrier(1)}
    bars.update({f"kv_full{s}@0": Barrier(2) for s in range(STAGES)})
    for r in RANKS:
        bars.update({f"o_done@{r}": Barrier(1)})
        bars.update({f"kv_empty{s}@{r}": Barrier(1) for s in range(STAGES)})
        bars.update({f"s_full{b}@{r}": Barrier(1) for b in range(SBUF)})
    progs = roles(n)
    pc = {r: 0 for r in progs}
    content = {}          # buffer -> tile it holds
    consumed = {}         # S buffer -> last tile the softmax read from it
    busy = {}             # buffer -> number of in-flight MMAs reading or writing it
    inflight = []         # issued MMAs, completed in order: (reads, writes)
    commits = []          # (barrier, number of MMAs issued before the commit)
    issued = completed = 0

    def check_write(buf, tile):
        assert busy.get(buf, 0) == 0, f"{buf} overwritten while an MMA uses it (tile {tile})"

    for _ in range(10 ** 6):
        runnable = []
        for r, prog in progs.items():
            if pc[r] < len(prog):
                a = prog[pc[r]]
                if a[0] != "wait" or bars[a[1]].done > a[2]:
                    runnable.append(r)
        if inflight:
            runnable.append("tensor_core")
        if not runnable:
            break
        r = rng.choice(runnable)
        if r == "tensor_core":
            reads, writes = inflight.pop(0)
            for buf, tile in writes:
                content[buf] = tile
            for buf, _ in reads + writes:
                busy[buf] -= 1
            completed += 1
            while commits and commits[0][1] <= completed:
                for name in commits.pop(0)[0]:
                    bars[name].arrive()
            continue
        a = progs[r][pc[r]]
        pc[r] += 1
        kind = a[0]
        if kind == "wait":
            # the waited completion index is a[2]; more than one further phase would alias
            assert bars[a[1]].done <= a[2] + 1, f"{r}: {a[1]} ran two phases ahead of completion {a[2]}"
        elif kind == "arrive":
            bars[a[1]].arrive()
        elif kind == "commit":
            commits.append((a[1], issued))
            while commits and commits[0][1] <= completed:
                for name in commits.pop(0)[0]:
                    bars[name].arrive()
        elif kind == "write":
            check_write(a[1], a[2])
            content[a[1]] = a[2]
        elif kind == "read":
            want = a[2] if not a[1].startswith("O") else n - 1
            assert content.get(a[1]) == want, f"{r} read {a[1]} holding {content.get(a[1])}, wanted {want}"
            consumed[a[1]] = a[2]
        elif kind == "issue":
            _, name, tile, reads, writes = a
            for buf, t in reads:
                want = t
                assert content.get(buf) == want, f"{name}({tile}) reads {buf} holding {content.get(buf)}"
            for buf, t in writes:
                if buf.startswith("O"):
                    assert content.get(buf) in (None, tile - 1, tile), f"PV({tile}) on {buf} of {content.get(buf)}"
                else:
                    check_write(buf, t)
                    if buf.startswith("S") and t >= SBUF:   # that CTA's softmax is done with the tile before
                        assert consumed.get(buf) == t - SBUF, f"S({t}) issued before {buf} of {t - SBUF} was read"
            for buf, _ in reads + writes:
                busy[buf] = busy.get(buf, 0) + 1
            inflight.append((reads, writes))
            issued += 1
    assert all(pc[r] == len(p) for r, p in progs.items()), f"deadlock: {pc}"


@pytest.mark.parametrize("n", list(range(1, 11)) + [17])
def test_protocol_under_random_interleavings(n):
    for seed in range(200):
        run(n, seed)


@pytest.mark.parametrize("drop", [
    ("loader0", "kv_empty"),   # a stage refilled while its P V may still run
    ("loader1", "kv_empty"),
    ("softmax0", "o_done"),    # P overwritten / O rescaled under a running P V
    ("softmax1", "o_done"),
    ("mma", "p_full"),         # P V issued before the softmax wrote P
    ("mma", "kv_full"),        # S issued before the loaders filled the stage
    ("softmax0", "s_full"),    # S read before the tensor core wrote it
    ("softmax1", "s_full"),
])
def test_model_catches_each_missing_wait(drop, monkeypatch):
    # the checks have teeth: removing any one kind of wait from a role breaks them
    role, bar = drop
    full = roles

    def mutated(n):
        r = full(n)
        r[role] = [a for a in r[role] if not (a[0] == "wait" and a[1].startswith(bar))]
        return r

    monkeypatch.setitem(globals(), "roles", mutated)
    with pytest.raises(AssertionError):
        for seed in range(300):
            run(9, seed)


def test_model_catches_a_count_of_one_arrival(monkeypatch):
    # rank 0's kv_full must wait for both CTAs' halves: with one arrival per
    # phase it completes on whichever CTA is first, and an MMA reads a half
    # that is not yet written
    orig = Barrier.__init__

    def one(self, count):
        orig(self, 1)

    monkeypatch.setattr(Barrier, "__init__", one)
    with pytest.raises(AssertionError):
        for seed in range(300):
            run(9, seed)

