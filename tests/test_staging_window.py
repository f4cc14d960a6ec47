"""Bounded staging window (back-pressure), host side, without a GPU.

The plan stages the remote rows through W slots of 256 rows: row block b (an
m-tile of a remote shard, in consumption order) lives in slot b % W, and the
producer may write block b only once every tile of block b - W has read its
rows.  These tests check the chunk rule such a plan uses, and -- by simulating
the persistent schedule exactly as the kernel walks it (tile order from the
library's own ag_gemm_tile_at; the local shard's tiles dealt round-robin, the
remote tiles handed out by a ticket counter in that order to whichever CTA
pairs are running) -- that a window of at least one swizzle group (group_m =
8 blocks) always finishes, also when fewer pairs are resident than were
launched, while a smaller window can stall for good.  A static deal of every
tile to pairs (pair p takes tiles p, p + pairs, ...) is simulated too: under
partial residency it can stall, which is why the kernel hands the remote
tiles out at run time.
"""
import pytest

from all_gather_gemm_chunked_gb300 import binding as B_


def test_bounded_chunk_rule():
    for R in list(range(1, 600)) + [1024, 2048, 3000, 4096, 4095, 6144, 10000]:
        c = B_.ag_gemm_choose_chunk_rows_bounded(R)
        assert R % c == 0 and 256 % c == 0, R
        c0 = B_.ag_gemm_choose_chunk_rows(R)
        if 256 % c0 == 0:
            assert c == c0, R
        else:
            # the largest power of two dividing R with at least 64 chunks
            best = max([d for d in (1, 2, 4, 8, 16, 32, 64, 128, 256)
                        if R % d == 0 and R // d >= 64] or [1])
            assert c == best, R
    assert B_.ag_gemm_choose_chunk_rows_bounded(3000) == 8
    assert B_.ag_gemm_choose_chunk_rows_bounded(4096) == 64


def _block_of(g, local):
    S, MT = g.n_shards, g.m_tiles

    def block(t):
        src, mt, _ = B_.ag_gemm_tile_at(g, local, t)
        pos = (src - local) % S
        return None if pos == 0 else (pos - 1) * MT + mt
    return [block(t) for t in range(g.tiles)]


def _simulate_tickets(g, local, W, resident, pairs=None, dealt=0):
    """True if every tile completes when `pairs` pairs are launched, `resident`
    of them run at once (a waiting pair starts when a running one exits), and
    each pair first computes the tiles dealt to it (pair k: tiles k, k + pairs,
    ... below `dealt`), then takes tiles from a ticket counter in schedule
    order, starting at `dealt` (a pair holds its tile until the tile's block
    is produced, and exits when the tickets run out).  Producer: blocks in
    order, block b once the NT tiles of block b - W have read their rows."""
    pairs = resident if pairs is None else pairs
    blocks = _block_of(g, local)
    nblocks = (g.n_shards - 1) * g.m_tiles
    produced, consumed = 0, [0] * nblocks
    nxt = list(range(pairs))             # next dealt tile per pair
    holding = {}                         # running pair -> drawn tile it holds
    running = list(range(min(resident, pairs)))
    waiting = list(range(len(running), pairs))
    ticket, done = dealt, 0
    while True:
        progress = False
        while produced < nblocks and (produced < W or consumed[produced - W] == g.n_tiles):
            produced += 1
            progress = True
        for p in list(running):
            while True:
                if nxt[p] < dealt:
                    t = nxt[p]
                elif p in holding:
                    t = holding[p]
                elif ticket < g.tiles:
                    t = holding[p] = ticket
                    ticket += 1
                    progress = True
                else:
                    running.remove(p)            # tickets exhausted: the pair exits
                    if waiting:
                        running.append(waiting.pop(0))
                    progress = True
                    break
                b = blocks[t]
                if b is not None and b >= produced:
                    break
                if b is not None:
                    consumed[b] += 1
                if nxt[p] < dealt:
                    nxt[p] += pairs
                else:
                    del holding[p]
                done += 1
                progress = True
        if done == g.tiles:
            return True
        if not progress:
            return False


def _simulate_static(g, local, W, pairs, resident):
    """The static deal: pair p takes tiles p, p + pairs, ...; only the first
    `resident` pairs run, a later pair starts when a running one has finished
    all of its tiles."""
    blocks = _block_of(g, local)
    nblocks = (g.n_shards - 1) * g.m_tiles
    produced, consumed = 0, [0] * nblocks
    nxt = list(range(min(pairs, g.tiles)))
    running = list(range(min(resident, len(nxt))))
    waiting = list(range(len(running), len(nxt)))
    done = 0
    while True:
        progress = False
        while produced < nblocks and (produced < W or consumed[produced - W] == g.n_tiles):
            produced += 1
            progress = True
        for p in list(running):
            while nxt[p] < g.tiles:
                b = blocks[nxt[p]]
                if b is not None and b >= produced:
                    break
                if b is not None:
                    consumed[b] += 1
                nxt[p] += pairs
                done += 1
                progress = True
            if nxt[p] >= g.tiles:
                running.remove(p)
                if waiting:
                    running.append(waiting.pop(0))
                progress = True
        if done == g.tiles:
            return True
        if not progress:
            return False


def _simulate(g, local, W, pairs):
    """True if every tile completes.  Producer: blocks in order, block b once
    the NT tiles of block b - W have read their rows.  Consumers: pair p takes
    tiles p, p + pairs, ... in order; a remote tile needs its block produced."""
    S, MT, NT = g.n_shards, g.m_tiles, g.n_tiles
    order = [B_.ag_gemm_tile_at(g, local, t) for t in range(g.tiles)]

    def block(tile):
        src, mt, _ = tile
        pos = (src - local) % S
        return None if pos == 0 else (pos - 1) * MT + mt

    nblocks = (S - 1) * MT
    produced, consumed = 0, [0] * nblocks
    nxt = list(range(min(pairs, g.tiles)))  # next tile index per pair
    done = 0
    while True:
        progress = False
        while produced < nblocks and (produced < W or consumed[produced - W] == NT):
            produced += 1
            progress = True
        for p in range(len(nxt)):
            while nxt[p] < g.tiles:
                b = block(order[nxt[p]])
                if b is not None and b >= produced:
                    break
                if b is not None:
                    consumed[b] += 1
                nxt[p] += pairs
                done += 1
                progress = True
        if done == g.tiles:
            return True
        if not progress:
            return False


@pytest.mark.parametrize("S,R,N", [(2, 4096, 4096), (4, 4096, 4096), (8, 1024, 4096),
                                   (3, 600, 392), (5, 2560, 1024), (3, 8 * 256 + 7, 768)])
def test_window_of_a_swizzle_group_always_finishes(S, R, N):
    g = B_.ag_gemm_geometry_of(S, S * R, 256, N, 0, 0)
    assert g.group_m == 8
    for W in (8, 9, 16, 17):
        for pairs in (1, 2, 7, 76):
            for local in {0, S - 1}:
                assert _simulate(g, local, W, pairs), (S, R, N, W, pairs, local)


@pytest.mark.parametrize("S,R,N", [(4, 4096, 4096), (8, 1024, 4096), (3, 600, 392),
                                   (5, 2560, 1024)])
def test_window_with_tickets_finishes_under_partial_residency(S, R, N):
    g = B_.ag_gemm_geometry_of(S, S * R, 256, N, 0, 0)
    for W in (8, 16):
        for resident in (1, 7, 38, 76):
            for local in {0, S - 1}:
                assert _simulate_tickets(g, local, W, resident), (S, R, N, W, resident, local)


@pytest.mark.parametrize("S,R,N", [(4, 4096, 4096), (8, 1024, 4096), (3, 600, 392),
                                   (5, 2560, 1024)])
def test_window_with_local_tiles_dealt_finishes_under_partial_residency(S, R, N):
    # the kernel deals the local shard's tiles (position 0: the first MT x NT
    # in schedule order, no rows to wait for, no credits) and draws the rest
    g = B_.ag_gemm_geometry_of(S, S * R, 256, N, 0, 0)
    for local in {0, S - 1}:
        blocks = _block_of(g, local)
        n_local = g.m_tiles * g.n_tiles
        assert all(b is None for b in blocks[:n_local])
        assert all(b is not None for b in blocks[n_local:])
        for W in (8, 16):
            for resident in (1, 7, 38, 76):
                assert _simulate_tickets(g, local, W, resident, pairs=76, dealt=n_local), \
                    (S, R, N, W, resident, local)


def test_static_deal_can_stall_under_partial_residency():
    # workload 4's shape with a window of 16 slots: 76 pairs launched, 7 resident
    g = B_.ag_gemm_geometry_of(4, 4 * 4096, 256, 4096, 0, 0)
    assert _simulate_static(g, 0, 16, 76, 76)
    assert not _simulate_static(g, 0, 16, 76, 7)
    assert _simulate_tickets(g, 0, 16, 7)
    assert _simulate_tickets(g, 0, 16, 7, pairs=76, dealt=g.m_tiles * g.n_tiles)
    # dealing one remote tile more is enough to stall
    assert not _simulate_tickets(g, 0, 16, 7, pairs=76, dealt=g.m_tiles * g.n_tiles + 76)


def test_window_below_a_swizzle_group_can_stall():
    g = B_.ag_gemm_geometry_of(2, 2 * 8 * 256, 256, 512, 0, 0)  # 8 m-tiles, 2 n-tiles
    assert g.m_tiles == 8 and g.n_tiles == 2
    # one pair walks the group m-fastest: it needs block 4 before block 0 is done
    assert not _simulate(g, 0, 4, 1)
    assert _simulate(g, 0, 8, 1)
    assert not _simulate_tickets(g, 0, 4, 1)
    assert _simulate_tickets(g, 0, 8, 1)
