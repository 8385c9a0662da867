"""Host-side model of the decode's work split and split-K bookkeeping.

The decode flattens the page-heads of all sequences -- (sequence, KV head,
page) items -- and cuts them into gridDim.x balanced contiguous CTA ranges,
each CTA range into kNW balanced contiguous warp ranges.  Inside a warp range
a maximal run of one (sequence, KV head) pair's items is a piece.  A piece
that does not cover its pair from the first page to the last becomes a record:
slot 1 if it is the last of two or more pieces of the warp's range, else slot
0.  A warp whose range is empty marks its slot-0 record empty.  The combine
rederives, from the lengths alone, the warps holding a pair's first and last
page-heads, takes the first warp's record (slot 1 unless the pair starts that
warp's range), then slot 0 of every later warp up to the last, skipping empty
records.

This model replays that arithmetic (restated from the kernel's description,
in Python) for many ragged batches and checks that each cut pair's records
are exactly the pieces that cover it, each page once and in order, and that
every record index stays inside the workspace the library sizes.  It needs no
GPU.
"""
import numpy as np
import pytest

PAGE = 16
NW = 4            # warps per CTA
CTAS_PER_SM = 3


def cta_start(c, W, N):
    q, rem = divmod(W, N)
    return c * q + min(c, rem)


def cta_of(r, W, N):
    q, rem = divmod(W, N)
    big = rem * (q + 1)
    return r // (q + 1) if r < big else rem + (r - big) // q


def warp_of_item(r, W, N):
    c = cta_of(r, W, N)
    r0 = cta_start(c, W, N)
    ln = cta_start(c + 1, W, N) - r0
    return c * NW + ((r - r0 + 1) * NW - 1) // ln


def simulate(lens, hkv, nsm):
    N = nsm * CTAS_PER_SM
    npg = [(L + PAGE - 1) // PAGE for L in lens]
    items = [(b, h, pg) for b, n in enumerate(npg) for h in range(hkv) for pg in range(n)]
    W = len(items)
    records = {}      # record index -> (b, h, first page, last page) or "empty"
    outputs = set()
    if W == 0:
        return
    for c in range(N):
        r0, r1 = cta_start(c, W, N), cta_start(c + 1, W, N)
        for w in range(NW):
            gw = c * NW + w
            wr0, wr1 = r0 + (r1 - r0) * w // NW, r0 + (r1 - r0) * (w + 1) // NW
            n = wr1 - wr0
            if n == 0:
                records[2 * gw] = "empty"
                continue
            i, nseg = 0, 0
            while i < n:
                b, h, page0 = items[wr0 + i]
                iend = min(n, i + (npg[b] - page0))
                nseg += 1
                last_page = page0 + (iend - i) - 1
                complete = page0 == 0 and last_page == npg[b] - 1
                slot = 1 if (iend == n and nseg > 1) else 0
                if complete:
                    outputs.add((b, h))
                else:
                    assert 2 * gw + slot not in records
                    records[2 * gw + slot] = (b, h, page0, last_page)
                i = iend
    before = 0
    for b, n in enumerate(npg):
        for h in range(hkv):
            if n == 0:
                continue
            # the combine's view: from the lengths alone
            p0 = before * hkv + h * n
            wf, wl = warp_of_item(p0, W, N), warp_of_item(p0 + n - 1, W, N)
            if wl == wf:
                assert (b, h) in outputs
                continue
            assert (b, h) not in outputs
            cf = wf // NW
            r0c, r1c = cta_start(cf, W, N), cta_start(cf + 1, W, N)
            wr0 = r0c + (r1c - r0c) * (wf - cf * NW) // NW
            first = 2 * wf + (1 if p0 > wr0 else 0)
            pages = []
            for c in range(wl - wf + 1):
                ri = first if c == 0 else 2 * (wf + c)
                assert ri < 2 * N * NW                   # inside the workspace's records
                rec = records[ri]
                if rec == "empty":
                    continue
                rb, rh, q0, q1 = rec
                assert (rb, rh) == (b, h)
                pages.extend(range(q0, q1 + 1))
            assert pages == list(range(n))               # each page once, in order
        before += n


@pytest.mark.parametrize("seed", range(40))
def test_records_tile_every_cut_pair(seed):
    rng = np.random.default_rng(seed)
    hkv = int(rng.choice([1, 2, 3, 4, 8, 16]))
    batch = int(rng.integers(1, 40))
    kind = seed % 4
    if kind == 0:
        lens = rng.integers(0, 300, batch)
    elif kind == 1:
        lens = rng.integers(0, 40, batch)                # fewer items than warps: empty warp ranges
    elif kind == 2:
        lens = np.exp(rng.uniform(np.log(1), np.log(20000), batch)).astype(int)
    else:
        lens = [int(rng.integers(1, 200000))]             # one long sequence over many CTAs
    nsm = int(rng.choice([4, 7, 152]))
    simulate([int(x) for x in lens], hkv, nsm)


def test_the_benchmark_shapes():
    simulate([8193] * 32, 8, 152)                         # 8K decode: 131,328 page-heads, 1824 warps
    simulate([131072] * 4, 8, 152)                        # 128K decode
    rng = np.random.default_rng(5)
    simulate(list(np.exp(rng.uniform(np.log(512), np.log(32768), 256)).astype(int) + 1), 8, 152)
    simulate([101, 258], 2, 152)                          # the tiny workload: most warps are empty


def test_empty_warps_lie_inside_cut_pairs_of_small_batches():
    # 48 page-heads over 1824 warps: most pairs are cut across warps with
    # empty ranges between them, the case the combine must skip
    simulate([101, 258], 2, 152)
    simulate([5, 3, 40], 1, 152)
