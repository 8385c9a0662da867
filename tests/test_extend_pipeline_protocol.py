"""Model check of the extend-attention kernel's synchronisation protocol (host only).

The kernel (csrc/extend_attention.cu) runs three roles in a CTA around
mbarriers: loader warps fill a three-stage K/V ring and write Q; one thread
issues the tensor-core MMAs (S = Q K^T into two S buffers, O += P V) and
commits each group to an mbarrier; softmax warps read S, rescale O and write P.
The tensor core finishes issued MMAs in order, asynchronously.  This model
replays each role's sequence of waits, arrivals, commits and buffer accesses,
in the kernel's order, under random interleavings, and checks:

- every wait targets the completion it means: the barrier has at most one
  more completed phase than the one waited for (else the parity would alias);
- no buffer is overwritten while an earlier user may still read it (K/V
  stages, S buffers, P, O), and every read sees the tile it expects;
- every interleaving finishes (no deadlock).
"""
import random

import pytest

STAGES, SBUF = 3, 2


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0  # done = completed phases

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


def roles(n):
    """The kernel's three roles as action lists (see the module docstring)."""
    loader = [("write", "Q", 0), ("arrive", "q_full")]
    for i in range(n):
        s = i % STAGES
        if i >= STAGES:
            loader.append(("wait", f"kv_empty{s}", i // STAGES - 1))
        loader += [("write", f"KV{s}", i), ("arrive", f"kv_full{s}")]
    mma = [("wait", "q_full", 0)]
    for i in range(n + 1):
        if i < n:
            s = i % STAGES
            mma += [("wait", f"kv_full{s}", i // STAGES),
                    ("issue", "S", i, [("Q", 0), (f"KV{s}", i)], [(f"S{i % SBUF}", i)]),
                    ("commit", f"s_full{i % SBUF}")]
        if i >= 1:
            pi = i - 1
            mma += [("wait", "p_full", pi),
                    ("issue", "PV", pi, [("P", pi), (f"KV{pi % STAGES}", pi)], [("O", pi)]),
                    ("commit", "o_done")]
            if pi + STAGES < n:
                mma.append(("commit", f"kv_empty{pi % STAGES}"))
    mma += [("commit", "drain"), ("wait", "drain", 0)]
    softmax = []
    for i in range(n):
        softmax += [("wait", f"s_full{i % SBUF}", i // SBUF), ("read", f"S{i % SBUF}", i)]
        if i >= 1:
            softmax += [("wait", "o_done", i - 1), ("write", "O", i)]   # the lazy rescale of O
        softmax += [("write", "P", i), ("arrive", "p_full")]
    softmax += [("wait", "o_done", n - 1), ("read", "O", n)]
    return {"loader": loader, "mma": mma, "softmax": softmax}


def run(n, seed):
    rng = random.Random(seed)
    bars = {name: Barrier(1) for name in ["q_full", "p_full", "o_done", "drain"] +
            [f"kv_full{s}" for s in range(STAGES)] + [f"kv_empty{s}" for s in range(STAGES)] +
            [f"s_full{b}" for b in range(SBUF)]}
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
                bars[commits.pop(0)[0]].arrive()
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
                bars[commits.pop(0)[0]].arrive()
        elif kind == "write":
            check_write(a[1], a[2])
            content[a[1]] = a[2]
        elif kind == "read":
            want = a[2] if a[1] != "O" else n - 1
            assert content.get(a[1]) == want, f"{r} read {a[1]} holding {content.get(a[1])}, wanted {want}"
            consumed[a[1]] = a[2]
        elif kind == "issue":
            _, name, tile, reads, writes = a
            for buf, t in reads:
                want = t
                assert content.get(buf) == want, f"{name}({tile}) reads {buf} holding {content.get(buf)}"
            for buf, t in writes:
                if buf == "O":
                    assert content.get("O") in (None, tile - 1, tile), f"PV({tile}) on O of {content.get('O')}"
                else:
                    check_write(buf, t)
                    if buf.startswith("S") and t >= SBUF:   # the softmax is done with the tile before
                        assert consumed.get(buf) == t - SBUF, f"S({t}) issued before {buf} of {t - SBUF} was read"
            for buf, _ in reads + writes:
                busy[buf] = busy.get(buf, 0) + 1
            inflight.append((reads, writes))
            issued += 1
    assert all(pc[r] == len(p) for r, p in progs.items()), f"deadlock: {pc}"


@pytest.mark.parametrize("n", list(range(1, 11)) + [17])
def test_protocol_under_random_interleavings(n):
    for seed in range(300):
        run(n, seed)


@pytest.mark.parametrize("drop", [
    ("loader", "kv_empty"),   # a stage refilled while its P V may still run
    ("softmax", "o_done"),    # P overwritten / O rescaled under a running P V
    ("mma", "p_full"),        # P V issued before the softmax wrote P
    ("mma", "kv_full"),       # S issued before the loaders filled the stage
    ("softmax", "s_full"),    # S read before the tensor core wrote it
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
            run(6, seed)
