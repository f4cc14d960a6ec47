"""Work items of the fused kernel, host side, without a GPU.

A pair's items are the whole tiles dealt to it round-robin (items k, k + P,
... below the dealt count), then, on the int8 path, items drawn from a
grid-wide ticket counter in schedule order -- the split parts of the last
round's tiles, whose last part waits for the earlier parts' partial sums.
The even CTA keeps up to two drawn items reserved ahead of the one it works
on.  This simulation checks that every item completes when only some of the
launched pairs are resident (the others start as resident pairs exit), for
the split counts the plan chooses, and that the item decode visits every
(tile, part) exactly once.  On the fp16 / bf16 path every item, split parts
included, is dealt (the parts add into zeroed C blocks and wait on no other
part): the two TMA producers of a pair then place item seq's k-blocks in the
shared ring after all earlier items' k-blocks, which is checked against a
plain running sum, and the zero tasks cover every tail tile's rows once.
"""
import pytest


def split_of(tiles, pairs, kb, i8=True):
    """The plan's rule: split the last round's tiles in two when they fill at
    most half of the pairs and a tile has at least 128 k-blocks (int8) or 32
    (fp16 / bf16)."""
    tail = tiles % pairs
    min_kb = 128 if i8 else 32
    return 2 if pairs >= 2 and tail and 2 * tail <= pairs and kb >= min_kb else 1


def items_of(tiles, pairs, kb, i8=True):
    s = split_of(tiles, pairs, kb, i8)
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


def part_blocks(kb, part, parts):
    """k-blocks [kb0, kb1) of part `part` of `parts` (the kernel's split)."""
    return kb * part // parts, kb * (part + 1) // parts


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
    assert split_of(256, 76, 64) == 1        # int8, short tiles: the hand-off would not pay
    assert split_of(228, 76, 128) == 1       # no partial round
    assert split_of(256, 76, 64, i8=False) == 2    # fp16 4096^3: parts add into C
    assert split_of(256, 76, 32, i8=False) == 2
    assert split_of(256, 76, 31, i8=False) == 1    # too short even so
    assert split_of(512, 76, 64, i8=False) == 1


def dealt_ring_block(seq, pair, pairs, full, split, kb, tiles):
    """The kernel's placement of a pair's dealt item seq in the k-block ring:
    KB per whole tile before it (the pair's whole tiles come first), then the
    k-blocks of the tail parts between its whole tiles and it."""
    n_whole = (full - pair + pairs - 1) // pairs if pair < full else 0
    g0 = min(seq, n_whole) * kb
    tail = tiles - full
    for j in range(n_whole, seq):
        i = pair + j * pairs
        part = (i - full) // tail
        b0, b1 = part_blocks(kb, part, split)
        g0 += b1 - b0
    return g0


@pytest.mark.parametrize("tiles,pairs,kb", [(256, 76, 64), (24, 76, 33), (8, 4, 40), (300, 76, 37),
                                            (7, 6, 64), (100, 76, 128)])
def test_dealt_ring_positions_follow_every_earlier_item(tiles, pairs, kb):
    full, work, decode = items_of(tiles, pairs, kb, i8=False)
    split = split_of(tiles, pairs, kb, i8=False)
    for pair in range(pairs):
        items = list(range(pair, work, pairs))   # every item dealt round-robin
        running = 0
        for seq, i in enumerate(items):
            assert dealt_ring_block(seq, pair, pairs, full, split, kb, tiles) == running
            t, part, parts = decode(i)
            b0, b1 = part_blocks(kb, part, parts)
            assert 0 <= b0 < b1 <= kb
            running += b1 - b0


@pytest.mark.parametrize("tiles,pairs", [(256, 76), (24, 76), (7, 6)])
def test_zero_tasks_cover_every_tail_tile_once(tiles, pairs):
    kb = 64
    full, work, decode = items_of(tiles, pairs, kb, i8=False)
    tail = tiles - full
    assert tail > 0
    tasks = tail * (256 // 32)                   # 32-row groups of a pair tile
    covered = [(full + tk // 8, (tk % 8) * 32) for tk in range(tasks)]
    assert len(set(covered)) == tasks
    assert {t for t, _ in covered} == set(range(full, tiles))
    # the parts that add into them are exactly the tail tiles' parts
    assert {decode(i)[0] for i in range(full, work)} == set(range(full, tiles))


def simulate_zeroing(tiles, pairs, kb, resident, warps=16):
    """The fp16 split tail's zero tasks under partial residency: each pair
    runs its dealt items in order; after its last whole tile each of its
    warps draws one zero task, before its first part each warp draws every
    task left and then waits until all tasks are done, and a pair with no
    part draws one per warp at its end.  A drawn task is done by its warp
    at once.  A resident pair that waits for tasks which no resident pair
    holds would never finish; a waiting pair leaves room for no other."""
    full, work, decode = items_of(tiles, pairs, kb, i8=False)
    tasks = (tiles - full) * 8
    state = {"next": 0, "done": 0}

    def draw(n):
        take = min(n, tasks - state["next"])
        state["next"] += take
        state["done"] += take               # done at once by the warp that drew it

    waiting, running = list(range(pairs)), []
    pos = {}
    while waiting and len(running) < resident:
        p = waiting.pop(0); running.append(p); pos[p] = 0
    finished = 0
    for _ in range(10 * work + 10 * pairs + 100):
        if not running:
            return finished == pairs
        p = running[0]
        items = list(range(p, work, pairs))
        i = pos[p]
        if i < len(items):
            _, part, parts = decode(items[i])
            if parts > 1:
                if i == 0 or decode(items[i - 1])[2] == 1:
                    draw(tasks)             # every task left, before the first wait
                if state["done"] < tasks:
                    return False            # would wait for tasks nobody running holds
            pos[p] = i + 1
            if parts == 1 and (i + 1 == len(items) or decode(items[i + 1])[2] > 1):
                draw(warps)                 # one task per warp after the last whole tile
            running.append(running.pop(0))
            continue
        if not items or decode(items[-1])[2] > 1:
            draw(0)                         # (its single draw came earlier, or none needed)
        running.pop(0)
        finished += 1
        if waiting:
            q = waiting.pop(0); running.append(q); pos[q] = 0
    return False


@pytest.mark.parametrize("tiles,kb", [(256, 64), (80, 32), (24, 64), (100, 37)])
def test_zero_tasks_never_wait_on_a_pair_that_has_not_started(tiles, kb):
    pairs = 76
    assert split_of(tiles, pairs, kb, i8=False) == 2
    for resident in (1, 2, 7, 38, 76):
        assert simulate_zeroing(tiles, pairs, kb, resident), (tiles, kb, resident)
