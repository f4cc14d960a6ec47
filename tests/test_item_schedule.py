"""Work items of the fused kernel, host side, without a GPU.

A pair's items are the whole tiles dealt to it round-robin (items k, k + P,
... below the dealt count), then items drawn from a grid-wide ticket counter
in schedule order -- the split parts of the last round's tiles, whose last
part waits for the earlier parts' partial sums.  The even CTA keeps up to two
drawn items reserved ahead of the one it works on.  This simulation checks
that every item completes when only some of the launched pairs are resident
(the others start as resident pairs exit), for the split counts the plan
chooses, and that the item decode visits every (tile, part) exactly once.
"""
import pytest


def split_of(tiles, pairs, kb):
    """The plan's rule: split the last round's tiles in two when they fill at
    most half of the pairs and a tile has at least 128 k-blocks."""
    tail = tiles % pairs
    return 2 if pairs >= 2 and tail and 2 * tail <= pairs and kb >= 128 else 1


def items_of(tiles, pairs, kb):
    s = split_of(tiles, pairs, kb)
    tail = tiles % pairs if s > 1 else 0
    full = tiles - tail
    work = full + tail * s

    def decode(i):
        if i < full:
            return i, 0, 1
        r = i - full
        part = r // tail
        return full + r - part * tail, part, s
    return full, work, decode


def simulate(tiles, pairs, kb, resident, ahead=2):
    full, work, decode = items_of(tiles, pairs, kb)
    done = set()
    ticket = full                      # drawn items start after the dealt ones
    queues = {}                        # running pair -> list of reserved items
    dealt_next = {}                    # pair -> next dealt item
    drawn_all = set()
    waiting = list(range(pairs))
    running = []

    def start(p):
        running.append(p)
        queues[p] = []
        dealt_next[p] = p

    while waiting and len(running) < resident:
        start(waiting.pop(0))
    steps = 0
    while len(done) < work:
        steps += 1
        if steps > 100 * work + 1000:
            return False
        progress = False
        for p in list(running):
            q = queues[p]
            # fill the queue: dealt items first, then tickets, up to 1 + ahead items
            while len(q) < 1 + ahead:
                if dealt_next[p] < full:
                    q.append(dealt_next[p])
                    dealt_next[p] += pairs
                elif p not in drawn_all:
                    if ticket < work:
                        q.append(ticket)
                        ticket += 1
                    else:
                        drawn_all.add(p)
                else:
                    break
            if not q:
                running.remove(p)           # the pair exits; a waiting one starts
                if waiting:
                    start(waiting.pop(0))
                progress = True
                continue
            t, part, parts = decode(q[0])
            if part == parts - 1 and parts > 1:
                # the last part waits for the earlier parts of its tile
                earlier = [i for i in range(full, work) if decode(i)[0] == t and decode(i)[1] < part]
                if not all(i in done for i in earlier):
                    continue
            done.add(q.pop(0))
            progress = True
        if not progress:
            return False
    return True


@pytest.mark.parametrize("tiles,kb", [(256, 128), (1024, 428), (28, 128), (104, 256), (96, 64),
                                      (3, 129), (77, 128)])
def test_every_item_completes_under_partial_residency(tiles, kb):
    pairs = 76
    for resident in (1, 2, 7, 38, 76):
        assert simulate(tiles, pairs, kb, resident), (tiles, kb, resident)


@pytest.mark.parametrize("tiles,pairs,kb", [(256, 76, 128), (1024, 76, 428), (8, 76, 130),
                                            (100, 76, 160), (500, 76, 128), (12, 4, 200)])
def test_item_decode_covers_every_tile_part_once(tiles, pairs, kb):
    full, work, decode = items_of(tiles, pairs, kb)
    seen = [decode(i) for i in range(work)]
    assert len(set((t, part) for t, part, _ in seen)) == work
    for t in range(tiles):
        parts = [s for tt, _, s in seen if tt == t]
        assert parts and all(s == len(parts) for s in parts)
    # the drawn items go part-major: every first part before any last part
    tail = [decode(i) for i in range(full, work)]
    firsts = [i for i, (t, part, s) in enumerate(tail) if part == 0]
    lasts = [i for i, (t, part, s) in enumerate(tail) if s > 1 and part == s - 1]
    assert not lasts or max(firsts) < min(lasts)


def test_split_rule():
    assert split_of(256, 76, 128) == 2       # 28 tiles left for 76 pairs
    assert split_of(1024, 76, 428) == 2      # 36 left (the int8 workload of 4 x 4096 rows)
    assert split_of(512, 76, 128) == 1       # 56 left: more than half of the pairs
    assert split_of(256, 76, 64) == 1        # short tiles: the split would not pay
    assert split_of(228, 76, 128) == 1       # no partial round
