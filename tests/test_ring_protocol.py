"""A model of the AdaLN kernel's row ring (host logic, no GPU): one producer
fills NS one-row stages in row order, compute warp w consumes rows
w, w + W, ... of the CTA's range, and the waits are mbarrier parity waits.
Random interleavings, with bulk copies completing in any order, check the
kernel's protocol -- a warp first waits until the producer has issued its
row, then waits on the stage's parity -- for stale reads and deadlock, and
show why the issued count is there: with the parity wait alone a warp can
take a stale row whenever the stage's previous row belongs to another warp
(NS != W) and has not landed yet."""
import random

import pytest


def _parity_passed(phases_done: int, parity: int) -> bool:
    """mbarrier try_wait.parity: true once the phase of that parity has
    completed, i.e. while the current (incomplete) phase has the other parity."""
    return (phases_done & 1) != parity


def run_ring(n_rows: int, W: int, NS: int, rng: random.Random, issued_count: bool, in_order: bool = False) -> int:
    """One random interleaving; returns the number of stale reads (a warp
    reading a stage whose data is not its row).  Raises on deadlock."""
    full = [0] * NS      # completed phases of each stage's "full" barrier
    empty = [0] * NS     # completed phases of each stage's "empty" barrier
    data = [None] * NS   # row held by each stage
    in_flight = []       # (stage, row) copies issued, not yet landed, in issue order
    issued = 0           # rows the producer has issued
    next_row = list(range(W))  # each warp's next row
    stale = 0
    while True:
        moves = []
        if issued < n_rows and _parity_passed(empty[issued % NS], ((issued // NS) & 1) ^ 1):
            moves.append(("produce", None))
        if in_flight:
            moves.append(("land", None))
        for w in range(W):
            i = next_row[w]
            if i >= n_rows or (issued_count and issued <= i):
                continue
            if _parity_passed(full[i % NS], (i // NS) & 1):
                moves.append(("consume", w))
        if not moves:
            break
        kind, w = rng.choice(moves)
        if kind == "produce":
            in_flight.append((issued % NS, issued))
            issued += 1
        elif kind == "land":
            st, row = in_flight.pop(0 if in_order else rng.randrange(len(in_flight)))
            data[st] = row
            full[st] += 1
        else:
            i = next_row[w]
            st = i % NS
            if data[st] != i:
                stale += 1
            empty[st] += 1
            next_row[w] = i + W
    if stale == 0 and not all(r >= n_rows for r in next_row):
        raise AssertionError("deadlock: a warp never got its row")
    return stale


SHAPES = [(8, 3), (8, 8), (8, 10), (8, 12), (14, 16), (16, 18), (16, 35)]


@pytest.mark.parametrize("W,NS", SHAPES)
def test_issued_count_then_parity_never_reads_a_stale_row(W, NS):
    rng = random.Random(W * 100 + NS)
    for _ in range(300):
        assert run_ring(3 * NS + 5, W, NS, rng, issued_count=True) == 0


def test_parity_alone_is_safe_only_with_in_order_landing_and_ns_at_least_w():
    rng = random.Random(1)
    for W, NS in [(8, 8), (8, 10), (16, 18)]:
        for _ in range(200):
            assert run_ring(3 * NS + 5, W, NS, rng, issued_count=False, in_order=True) == 0


@pytest.mark.parametrize("W,NS,in_order", [(8, 10, False), (16, 18, False), (8, 6, True)])
def test_parity_alone_can_read_a_stale_row(W, NS, in_order):
    rng = random.Random(W * 1000 + NS)
    assert any(run_ring(3 * NS + 5, W, NS, rng, issued_count=False, in_order=in_order) > 0 for _ in range(3000))


def run_broadcast_ring(n_chunks: int, W: int, NS: int, rng: random.Random) -> int:
    """The norm/RoPE kernel's ring: every compute warp reads every chunk (its
    own rows of it) in chunk order, the stage's "empty" barrier completes when
    all W warps have arrived, and the waits are parity waits alone.  A warp
    waiting for chunk c has itself consumed chunk c - NS of the same stage, so
    that fill has landed whatever order the copies complete in.  Returns the
    number of stale reads."""
    full = [0] * NS
    empty_arrivals = [0] * NS
    data = [None] * NS
    in_flight = []
    issued = 0
    next_chunk = [0] * W
    stale = 0
    while True:
        moves = []
        if issued < n_chunks and _parity_passed(empty_arrivals[issued % NS] // W, ((issued // NS) & 1) ^ 1):
            moves.append(("produce", None))
        if in_flight:
            moves.append(("land", None))
        for w in range(W):
            c = next_chunk[w]
            if c < n_chunks and _parity_passed(full[c % NS], (c // NS) & 1):
                moves.append(("consume", w))
        if not moves:
            break
        kind, w = rng.choice(moves)
        if kind == "produce":
            in_flight.append((issued % NS, issued))
            issued += 1
        elif kind == "land":
            st, c = in_flight.pop(rng.randrange(len(in_flight)))
            data[st] = c
            full[st] += 1
        else:
            c = next_chunk[w]
            stale += data[c % NS] != c
            empty_arrivals[c % NS] += 1
            next_chunk[w] = c + 1
    assert all(c >= n_chunks for c in next_chunk), "deadlock"
    return stale


@pytest.mark.parametrize("W,NS", [(8, 2), (8, 3), (4, 3)])
def test_broadcast_ring_of_the_norm_kernel_needs_no_issued_count(W, NS):
    rng = random.Random(W * 10 + NS)
    for _ in range(300):
        assert run_broadcast_ring(4 * NS + 3, W, NS, rng) == 0
