"""A model of the one-query-tile attention pipeline's synchronisation (host
logic, no GPU), as the persistent kernel runs it over a stream of units (the
single-CTA-per-unit kernel is the one-unit case).

Roles: a producer fills an NSTAGE ring in the order K0, K1, K2, then K_{J+3},
V_J; two MMA-issuing threads take even / odd key tiles (thread p issues
O += P_J V_J and then S_{J+3} = Q K_{J+3}^T into score buffer (J+1) mod 2);
the softmax reads S_J, publishes P_J into a single P buffer once
O += P_{J-1} V_{J-1} has completed, writes the next unit's Q once the current
unit's last score tile is read, and reads O at each unit's end.  mbarrier
waits are parity waits (pass iff completed phases % 2 != parity); a
thread's MMAs complete in issue order only where they share an accumulator,
and its commits once all it issued before them completed; bulk copies
complete in any order.  Checked in every interleaving: every product reads
the stage, score buffer, P and Q it was meant to, the first P V of a unit
overwrites O only after the previous epilogue read it, nothing deadlocks.

The Q hand-off is a count of written query rows that an MMA thread waits on
before the first Q K^T of a unit.  The model also runs the hand-off it
replaced, a parity barrier, and finds the failure it had: an MMA thread that
skips a one-tile unit can no longer tell unit k's Q from unit k - 2's.

The padding warp (one unit per CTA) zeroes the V rows past kv_len of the key
tile that straddles it: it waits for the producer's flag that the tile's V
load is issued, then for the stage's phase, and the tile's P V waits for it.
Without the flag the phase wait could pass on an older fill of the stage.

run_two_tile models the two-tile kernel (one MMA-issuing thread, NQ query
tiles sharing each K/V tile, P_q written over S_q): the issuer's wait for
O_q += P_q V before the next S_q is what keeps S_q from overwriting an unread
P_q, since the two products write different accumulators.

run_wide models the head-dim-256 kernel (two score buffers, P over its
buffer, K/V in half tiles, O in two halves): besides the checks above, it
shows that its epilogue needs the one-shot drain wait, because a parity wait
on the last product can pass while the product before it is still pending."""
import random

import pytest


def take_tensor_op(queue, rng):
    """Removes and returns one tensor-core operation of a thread that may
    complete next: MMAs on the same accumulator complete in issue order, others
    in any order, and a commit (an mbarrier arrive once everything the thread
    issued before it has completed) only when nothing earlier is pending."""
    ready = []
    seen = set()
    for k, op in enumerate(queue):
        if op[0] == "commit":
            if k == 0:
                ready.append(k)
            continue
        if op[-1] not in seen:
            ready.append(k)
        seen.add(op[-1])
    return queue.pop(rng.choice(ready))


class Bar:
    """An mbarrier with an arrival count, counting completed phases."""

    def __init__(self, count=1):
        self.count, self.pending, self.done = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def ok(self, parity):
        return (self.done & 1) != parity


def run_pipe(units, seed, nstage, q_handoff="count", pad_tile=None, pad_flag=True):
    """One random interleaving over units of the given key-tile counts (0 =
    a unit with no key tile, which only writes zero rows and joins no stream).
    pad_tile: (one unit only) the key tile that straddles kv_len, whose V rows
    past kv_len a padding warp zeroes before that tile's P V; it first waits
    for the producer's flag that the tile's V load is issued (pad_flag), then
    for the stage's phase.  Returns the list of protocol violations."""
    rng = random.Random(seed)
    tiles = []   # (unit seq, tile index in unit) of each stream tile J
    seq = 0
    for n in units:
        if n > 0:
            tiles.extend((seq, j) for j in range(n))
            seq += 1
    n_units = seq
    N = len(tiles)
    kv_full = [Bar() for _ in range(nstage)]
    kv_empty = [Bar() for _ in range(nstage)]
    s_full, s_read = [Bar(), Bar()], [Bar(), Bar()]
    p_ready, pv_done = [Bar(), Bar()], [Bar(), Bar()]
    q_full = Bar()
    v_clean = Bar()
    st = {"q_ready": 0, "Q": None, "S": [None, None], "P": None, "O": None, "O_read": True,
          "stage": [None] * nstage, "pad_issued": False, "zeroed": None}
    queues = {0: [], 1: []}   # tensor-core operations of each MMA thread, in issue order
    copies = []               # bulk copies in flight: (stage, contents)
    errors = []

    def load_of_v(J):
        return min(J + 4, N) + J

    def load_of_k(J):
        return J if J < 3 else 2 * J - 3

    def buf_parity(J):        # tile J is use J // 2 of buffer J % 2
        return (J >> 1) & 1

    def producer():
        order = [("K", j) for j in range(min(3, N))]
        for J in range(N):
            if J + 3 < N:
                order.append(("K", J + 3))
            order.append(("V", J))
        for ld, what in enumerate(order):
            sidx, ph = ld % nstage, (ld // nstage) & 1
            yield lambda sidx=sidx, ph=ph: kv_empty[sidx].ok(ph ^ 1)
            copies.append((sidx, what))
            if what == ("V", pad_tile):
                st["pad_issued"] = True

    def pad_warp():
        ld = load_of_v(pad_tile)
        sidx, ph = ld % nstage, (ld // nstage) & 1
        if pad_flag:
            yield lambda: st["pad_issued"]
        yield lambda: kv_full[sidx].ok(ph)
        if st["stage"][sidx] != ("V", pad_tile):
            errors.append(f"padding warp zeroes stage {sidx} holding {st['stage'][sidx]}, not V of tile {pad_tile}")
        st["zeroed"] = pad_tile
        v_clean.arrive()

    def mma(p):
        if N <= p:
            return
        q_seq = [-1]

        def issue_qk(J):
            useq = tiles[J][0]
            if useq != q_seq[0]:
                if q_handoff == "count":
                    yield lambda: st["q_ready"] >= useq + 1
                else:
                    yield lambda: q_full.ok(useq & 1)
                q_seq[0] = useq
            ld = load_of_k(J)
            sidx, ph = ld % nstage, (ld // nstage) & 1
            yield lambda: kv_full[sidx].ok(ph)
            if J >= 2:
                yield lambda: s_read[J & 1].ok(buf_parity(J - 2))
            queues[p].extend([("qk", J, sidx, ("S", J & 1)), ("commit", s_full[J & 1]), ("commit", kv_empty[sidx])])

        yield from issue_qk(p)
        if p == 1 and N > 2:
            yield from issue_qk(2)
        for J in range(p, N, 2):
            ld = load_of_v(J)
            sidx, ph = ld % nstage, (ld // nstage) & 1
            yield lambda: kv_full[sidx].ok(ph)
            yield lambda: p_ready[p].ok(buf_parity(J))
            if J == pad_tile:
                yield lambda: v_clean.ok(0)
            queues[p].extend([("pv", J, sidx, ("O",)), ("commit", pv_done[p]), ("commit", kv_empty[sidx])])
            if J + 3 < N:
                yield from issue_qk(J + 3)

    def write_q(useq):
        st["Q"] = useq
        if q_handoff == "count":
            st["q_ready"] += 1
        else:
            q_full.arrive()

    def softmax():
        J = 0
        if N:
            write_q(0)
        useq = 0
        for n in units:
            if n == 0:
                continue
            for j in range(n):
                yield lambda: s_full[J & 1].ok(buf_parity(J))
                if st["S"][J & 1] != J:
                    errors.append(f"softmax reads score buffer {J & 1} holding tile {st['S'][J & 1]} for tile {J}")
                if j == n - 1 and useq + 1 < n_units:
                    write_q(useq + 1)
                s_read[J & 1].arrive()
                if J > 0:
                    yield lambda: pv_done[(J - 1) & 1].ok(buf_parity(J - 1))
                st["P"] = J
                p_ready[J & 1].arrive()
                J += 1
            yield lambda: pv_done[(J - 1) & 1].ok(buf_parity(J - 1))
            if st["O"] != (useq, n):
                errors.append(f"epilogue of unit {useq} reads O {st['O']}")
            st["O_read"] = True
            useq += 1

    def execute(p):
        op = take_tensor_op(queues[p], rng)
        if op[0] == "commit":
            op[1].arrive()
        elif op[0] == "qk":
            J, sidx = op[1], op[2]
            if st["stage"][sidx] != ("K", J):
                errors.append(f"Q K^T of tile {J} reads stage {sidx} holding {st['stage'][sidx]}")
            if st["Q"] != tiles[J][0]:
                errors.append(f"Q K^T of tile {J} (unit {tiles[J][0]}) reads the Q of unit {st['Q']}")
            st["S"][J & 1] = J
        else:
            J, sidx = op[1], op[2]
            if st["stage"][sidx] != ("V", J):
                errors.append(f"P V of tile {J} reads stage {sidx} holding {st['stage'][sidx]}")
            if st["P"] != J:
                errors.append(f"P V of tile {J} reads P of tile {st['P']}")
            if J == pad_tile and st["zeroed"] != J:
                errors.append(f"P V of tile {J} reads V before its padding rows were zeroed")
            useq, j = tiles[J]
            if j == 0:
                if not st["O_read"]:
                    errors.append(f"P V of tile {J} overwrites O before the epilogue read it")
                st["O"], st["O_read"] = (useq, 1), False
            else:
                if st["O"] != (useq, j):
                    errors.append(f"P V of tile {J} accumulates onto O {st['O']}")
                st["O"] = (useq, j + 1)

    roles = {"producer": producer(), "mma0": mma(0), "mma1": mma(1), "softmax": softmax()}
    if pad_tile is not None:
        assert len(units) == 1 and 0 <= pad_tile < units[0]
        roles["pad"] = pad_warp()
    waits = {}
    for name in list(roles):
        try:
            waits[name] = next(roles[name])
        except StopIteration:
            del roles[name]
    while roles or queues[0] or queues[1] or copies:
        moves = [("role", r) for r in roles if waits[r]()]
        moves += [("tensor", p) for p in (0, 1) if queues[p]]
        moves += [("copy", i) for i in range(len(copies))]
        if not moves:
            return [f"deadlock: {sorted(roles)} waiting"]
        kind, x = rng.choice(moves)
        if kind == "role":
            try:
                waits[x] = roles[x].send(None)
            except StopIteration:
                del roles[x]
        elif kind == "tensor":
            execute(x)
        else:
            sidx, what = copies.pop(x)
            st["stage"][sidx] = what
            kv_full[sidx].arrive()
        if errors:
            return errors
    return errors


def _random_units(rng):
    return [rng.choice([0, 1, 1, 2, 3, 5]) for _ in range(rng.randint(1, 7))]


@pytest.mark.parametrize("nstage", [4, 7, 12])
def test_count_handoff_pipeline_is_clean(nstage):
    rng = random.Random(nstage)
    for trial in range(400):
        units = _random_units(rng)
        assert run_pipe(units, trial, nstage) == [], f"units {units}, seed {trial}"


@pytest.mark.parametrize("n", [1, 2, 3, 8, 40])
def test_single_unit_pipeline_is_clean(n):
    # the default kernel: one unit per CTA
    for trial in range(100):
        assert run_pipe([n], trial, 7) == []


def test_parity_handoff_of_q_can_alias():
    rng = random.Random(7)
    failures = 0
    for trial in range(1500):
        failures += bool(run_pipe(_random_units(rng), trial, 7, q_handoff="parity"))
    assert failures > 0


@pytest.mark.parametrize("n", [1, 3, 9, 40])
def test_padding_warp_zeroes_the_right_tile_before_its_product(n):
    for trial in range(60):
        for pad in sorted({0, n // 2, n - 1}):
            assert run_pipe([n], trial, 7, pad_tile=pad) == [], f"n {n}, pad tile {pad}, seed {trial}"


def test_padding_warp_without_the_issue_flag_can_take_an_older_fill():
    # a phase wait counted from the kernel's start alone: the stage may pass
    # on a fill two rounds older, or be empty, when the padding tile's V is a
    # later fill of its stage
    bad = sum(bool(run_pipe([40], trial, 7, pad_tile=20, pad_flag=False)) for trial in range(200))
    assert bad > 0


def run_two_tile(n_tiles, NQ, nstage, seed, pad_tile=None, wait_pv_before_s=True):
    """One random interleaving of the two-tile kernel (attn_fwd): NQ query
    tiles share each K/V tile; the producer loads Q once, then K_j, V_j into
    an nstage ring; one MMA-issuing thread, per key tile j, waits for K_j and,
    per query tile q, for O_q += P_q V_{j-1} to complete (P_q lives over S_q)
    before S_q = Q_q K_j^T, then waits for V_j and each P_q before
    O_q += P_q V_j; softmax q waits for S_q, may rescale O_q (after waiting for
    the previous P V of its tile, which skips phases of that barrier), writes
    P_q over S_q and publishes it; the epilogue waits for the last P V.
    Returns the list of protocol violations."""
    rng = random.Random(seed)
    q_full = Bar()
    kv_full = [Bar() for _ in range(nstage)]
    kv_empty = [Bar() for _ in range(nstage)]
    s_full = [Bar() for _ in range(NQ)]
    p_ready = [Bar() for _ in range(NQ)]
    pv_done = [Bar() for _ in range(NQ)]
    v_clean = Bar()
    st = {"Q": False, "stage": [None] * nstage, "S": [None] * NQ, "P": [None] * NQ, "O": [0] * NQ,
          "pad_issued": False, "zeroed": None}
    queue = []
    copies = []
    errors = []

    def producer():
        copies.append(("Q", None))
        for ld in range(2 * n_tiles):
            sidx, ph = ld % nstage, (ld // nstage) & 1
            yield lambda sidx=sidx, ph=ph: kv_empty[sidx].ok(ph ^ 1)
            what = ("K" if ld % 2 == 0 else "V", ld // 2)
            copies.append((sidx, what))
            if what == ("V", pad_tile):
                st["pad_issued"] = True

    def pad_warp():
        ld = 2 * pad_tile + 1
        sidx, ph = ld % nstage, (ld // nstage) & 1
        yield lambda: st["pad_issued"]
        yield lambda: kv_full[sidx].ok(ph)
        if st["stage"][sidx] != ("V", pad_tile):
            errors.append(f"padding warp zeroes stage {sidx} holding {st['stage'][sidx]}")
        st["zeroed"] = pad_tile
        v_clean.arrive()

    def mma():
        yield lambda: q_full.ok(0)
        for j in range(n_tiles):
            sk, phk = (2 * j) % nstage, ((2 * j) // nstage) & 1
            yield lambda: kv_full[sk].ok(phk)
            for q in range(NQ):
                if j > 0 and wait_pv_before_s:
                    yield lambda q=q: pv_done[q].ok((j - 1) & 1)
                queue.extend([("qk", q, j, sk, ("S", q)), ("commit", s_full[q])])
            queue.append(("commit", kv_empty[sk]))
            sv, phv = (2 * j + 1) % nstage, ((2 * j + 1) // nstage) & 1
            yield lambda: kv_full[sv].ok(phv)
            if j == pad_tile:
                yield lambda: v_clean.ok(0)
            for q in range(NQ):
                yield lambda q=q: p_ready[q].ok(j & 1)
                queue.extend([("pv", q, j, sv, ("O", q)), ("commit", pv_done[q])])
            queue.append(("commit", kv_empty[sv]))

    def softmax(q):
        for j in range(n_tiles):
            yield lambda: s_full[q].ok(j & 1)
            if st["S"][q] != j:
                errors.append(f"softmax {q} reads S holding tile {st['S'][q]} for tile {j}")
            if j > 0 and rng.random() < 0.5:   # the running max grew: rescale O_q
                yield lambda: pv_done[q].ok((j - 1) & 1)
                if st["O"][q] != j:
                    errors.append(f"softmax {q} rescales O holding {st['O'][q]} tiles at tile {j}")
            st["P"][q] = j
            st["S"][q] = None   # P is written over S
            p_ready[q].arrive()
        if n_tiles:
            yield lambda: pv_done[q].ok((n_tiles - 1) & 1)
            if st["O"][q] != n_tiles:
                errors.append(f"epilogue {q} reads O holding {st['O'][q]} of {n_tiles} tiles")

    def execute():
        op = take_tensor_op(queue, rng)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, q, j, sidx, _ = op
        if kind == "qk":
            if not st["Q"]:
                errors.append(f"S_{q} of tile {j} reads Q before it landed")
            if st["stage"][sidx] != ("K", j):
                errors.append(f"S_{q} of tile {j} reads stage {sidx} holding {st['stage'][sidx]}")
            if st["P"][q] is not None and st["O"][q] != st["P"][q] + 1:
                errors.append(f"S_{q} of tile {j} overwrites P of tile {st['P'][q]} before O += P V read it")
            st["S"][q] = j
        else:
            if st["stage"][sidx] != ("V", j):
                errors.append(f"O_{q} += P V of tile {j} reads stage {sidx} holding {st['stage'][sidx]}")
            if j == pad_tile and st["zeroed"] != j:
                errors.append(f"O_{q} += P V of tile {j} reads V before its padding rows were zeroed")
            if st["P"][q] != j or st["O"][q] != j:
                errors.append(f"O_{q} += P V of tile {j} reads P {st['P'][q]} onto O of {st['O'][q]} tiles")
            st["O"][q] = j + 1

    roles = {"producer": producer(), "mma": mma()}
    roles.update({f"softmax{q}": softmax(q) for q in range(NQ)})
    if pad_tile is not None:
        roles["pad"] = pad_warp()
    waits = {}
    for name in list(roles):
        try:
            waits[name] = next(roles[name])
        except StopIteration:
            del roles[name]
    while roles or queue or copies:
        moves = [("role", r) for r in roles if waits[r]()]
        if queue:
            moves.append(("tensor", None))
        moves += [("copy", i) for i in range(len(copies))]
        if not moves:
            return [f"deadlock: {sorted(roles)} waiting"]
        kind, x = rng.choice(moves)
        if kind == "role":
            try:
                waits[x] = roles[x].send(None)
            except StopIteration:
                del roles[x]
        elif kind == "tensor":
            execute()
        else:
            sidx, what = copies.pop(x)
            if sidx == "Q":
                st["Q"] = True
                q_full.arrive()
            else:
                st["stage"][sidx] = what
                kv_full[sidx].arrive()
        if errors:
            return errors
    return errors


@pytest.mark.parametrize("NQ,nstage", [(1, 2), (1, 4), (2, 4), (2, 8), (1, 2)])
def test_two_tile_kernel_protocol_is_clean(NQ, nstage):
    for n in (1, 2, 5, 16):
        for trial in range(60):
            pad = None if trial % 3 == 0 else trial % n
            assert run_two_tile(n, NQ, nstage, trial, pad_tile=pad) == [], f"n {n}, pad {pad}, seed {trial}"


def test_two_tile_kernel_needs_the_wait_before_the_next_score_product():
    bad = sum(bool(run_two_tile(8, 2, 4, trial, wait_pv_before_s=False)) for trial in range(300))
    assert bad > 0


def run_separate_p(n_tiles, nstage, seed, pad_tile=None, s_read_wait=True):
    """One random interleaving of the two-CTA kernel's head-dim-64 form
    (attn_fwd, one query tile, P in a tensor-memory buffer of its own): the
    producer loads Q, then K_j, V_j into an nstage ring; the MMA thread issues
    S = Q K_0^T, then per key tile j: S = Q K_{j+1}^T once K_{j+1} has landed
    and the softmax has read S_j out (s_read), then O += P_j V_j once V_j has
    landed and P_j is published.  The softmax per tile waits for S_j, may
    rescale O (after the previous P V), arrives s_read, waits for the previous
    P V before writing P_j over the P buffer, publishes it; the epilogue waits
    for the last P V.  s_read_wait=False drops the MMA thread's s_read wait
    (a planted mistake).  Returns the list of protocol violations."""
    rng = random.Random(seed)
    q_full = Bar()
    kv_full = [Bar() for _ in range(nstage)]
    kv_empty = [Bar() for _ in range(nstage)]
    s_full, s_read, p_ready, pv_done, v_clean = Bar(), Bar(), Bar(), Bar(), Bar()
    st = {"Q": False, "stage": [None] * nstage, "S": None, "P": None, "O": 0, "pad_issued": False,
          "zeroed": None}
    queue, copies, errors = [], [], []

    def producer():
        copies.append(("Q", None))
        for ld in range(2 * n_tiles):
            sidx, ph = ld % nstage, (ld // nstage) & 1
            yield lambda sidx=sidx, ph=ph: kv_empty[sidx].ok(ph ^ 1)
            what = ("K" if ld % 2 == 0 else "V", ld // 2)
            copies.append((sidx, what))
            if what == ("V", pad_tile):
                st["pad_issued"] = True

    def pad_warp():
        ld = 2 * pad_tile + 1
        sidx, ph = ld % nstage, (ld // nstage) & 1
        yield lambda: st["pad_issued"]
        yield lambda: kv_full[sidx].ok(ph)
        if st["stage"][sidx] != ("V", pad_tile):
            errors.append(f"padding warp zeroes stage {sidx} holding {st['stage'][sidx]}")
        st["zeroed"] = pad_tile
        v_clean.arrive()

    def mma():
        yield lambda: q_full.ok(0)

        def qk(j):
            sk, phk = (2 * j) % nstage, ((2 * j) // nstage) & 1
            yield lambda: kv_full[sk].ok(phk)
            if j > 0 and s_read_wait:
                yield lambda: s_read.ok((j - 1) & 1)
            queue.extend([("qk", j, sk), ("commit", s_full), ("commit", kv_empty[sk])])

        if n_tiles:
            yield from qk(0)
        for j in range(n_tiles):
            if j + 1 < n_tiles:
                yield from qk(j + 1)
            sv, phv = (2 * j + 1) % nstage, ((2 * j + 1) // nstage) & 1
            yield lambda: kv_full[sv].ok(phv)
            if j == pad_tile:
                yield lambda: v_clean.ok(0)
            yield lambda: p_ready.ok(j & 1)
            queue.extend([("pv", j, sv), ("commit", pv_done), ("commit", kv_empty[sv])])

    def softmax():
        for j in range(n_tiles):
            yield lambda: s_full.ok(j & 1)
            if st["S"] != j:
                errors.append(f"softmax reads S holding {st['S']} for tile {j}")
            if j > 0 and rng.random() < 0.5:   # the running max grew: rescale O
                yield lambda: pv_done.ok((j - 1) & 1)
                if st["O"] != j:
                    errors.append(f"softmax rescales O holding {st['O']} tiles at tile {j}")
            st["S"] = ("read", j)
            s_read.arrive()
            if j > 0:
                yield lambda: pv_done.ok((j - 1) & 1)
            if st["O"] != j:
                errors.append(f"softmax writes P of tile {j} before O += P V of tile {j - 1} read the buffer")
            st["P"] = j
            p_ready.arrive()
        if n_tiles:
            yield lambda: pv_done.ok((n_tiles - 1) & 1)
            if st["O"] != n_tiles:
                errors.append(f"epilogue reads O holding {st['O']} of {n_tiles} tiles")

    def execute():
        op = take_tensor_op(queue, rng)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, j, sidx = op
        if kind == "qk":
            if not st["Q"]:
                errors.append(f"S of tile {j} reads Q before it landed")
            if st["stage"][sidx] != ("K", j):
                errors.append(f"S of tile {j} reads stage {sidx} holding {st['stage'][sidx]}")
            if isinstance(st["S"], int):
                errors.append(f"S of tile {j} overwrites unread scores of tile {st['S']}")
            st["S"] = j
        else:
            if st["stage"][sidx] != ("V", j):
                errors.append(f"O += P V of tile {j} reads stage {sidx} holding {st['stage'][sidx]}")
            if j == pad_tile and st["zeroed"] != j:
                errors.append(f"O += P V of tile {j} reads V before its padding rows were zeroed")
            if st["P"] != j or st["O"] != j:
                errors.append(f"O += P V of tile {j} reads P {st['P']} onto O of {st['O']} tiles")
            st["O"] = j + 1

    roles = {"producer": producer(), "mma": mma(), "softmax": softmax()}
    if pad_tile is not None:
        roles["pad"] = pad_warp()
    waits = {}
    for name in list(roles):
        try:
            waits[name] = next(roles[name])
        except StopIteration:
            del roles[name]
    while roles or queue or copies:
        moves = [("role", r) for r in roles if waits[r]()]
        if queue:
            moves.append(("tensor", None))
        moves += [("copy", i) for i in range(len(copies))]
        if not moves:
            return [f"deadlock: {sorted(roles)} waiting"]
        kind, x = rng.choice(moves)
        if kind == "role":
            try:
                waits[x] = roles[x].send(None)
            except StopIteration:
                del roles[x]
        elif kind == "tensor":
            execute()
        else:
            sidx, what = copies.pop(x)
            if sidx == "Q":
                st["Q"] = True
                q_full.arrive()
            else:
                st["stage"][sidx] = what
                kv_full[sidx].arrive()
        if errors:
            return errors
    return errors


@pytest.mark.parametrize("nstage", [3, 4, 6])
def test_separate_p_protocol_is_clean(nstage):
    for n in (1, 2, 3, 5, 16):
        for trial in range(80):
            pad = None if trial % 3 == 0 else trial % n
            assert run_separate_p(n, nstage, trial, pad_tile=pad) == [], f"n {n}, pad {pad}, seed {trial}"


def test_separate_p_needs_the_scores_read_wait():
    bad = sum(bool(run_separate_p(8, 4, trial, s_read_wait=False)) for trial in range(300))
    assert bad > 0


def run_wide(n_tiles, nstage, seed, pad_tile=None, epilogue="drain"):
    """One random interleaving of the head-dim-256 kernel (attn_wide): score
    buffers S_0, S_1 (tile j in S_{j mod 2}, P_j written over it), O in two
    128-channel halves, Q loaded once; the producer fills an nstage ring of
    half tiles in the order K_0, K_1, then V_j, K_{j+2} (two halves each);
    one MMA thread issues S_0 = Q K_0^T and S_1 = Q K_1^T, then per tile j
    waits for P_j, issues O_h += P_j V_j[h] for h = 0, 1, commits pv_done,
    and (if j + 2 < n) waits for that product before S_{j mod 2} =
    Q K_{j+2}^T; the softmax waits for S_j, may rescale O (after waiting for
    the previous product), writes P_j over S_j and publishes it.  The
    epilogue waits for the MMA thread's one-shot drain commit ("drain") or, as
    a parity wait on pv_done for the last tile ("parity"), which two pending
    products can alias.  Returns the list of protocol violations."""
    rng = random.Random(seed)
    q_full, drain, v_clean = Bar(), Bar(), Bar()
    kv_full = [Bar() for _ in range(nstage)]
    kv_empty = [Bar() for _ in range(nstage)]
    s_full, p_ready = [Bar(), Bar()], [Bar(), Bar()]
    pv_done = Bar()
    st = {"Q": False, "stage": [None] * nstage, "S": [None, None], "P": [None, None], "O": [0, 0],
          "pad_issued": False, "zeroed": None}
    queue, copies, errors = [], [], []
    n_lead = min(n_tiles, 2)

    def ld_v(j):
        return 2 * n_lead + 2 * j + 2 * max(0, min(j, n_tiles - 2))

    def ld_k(j):
        return 2 * j if j < 2 else ld_v(j - 2) + 2

    def producer():
        copies.append(("Q", None))
        order = [("K", j, h) for j in range(n_lead) for h in (0, 1)]
        for j in range(n_tiles):
            order += [("V", j, 0), ("V", j, 1)]
            if j + 2 < n_tiles:
                order += [("K", j + 2, 0), ("K", j + 2, 1)]
        for pos, what in enumerate(order):
            assert pos == (ld_k(what[1]) if what[0] == "K" else ld_v(what[1])) + what[2]
            sidx, ph = pos % nstage, (pos // nstage) & 1
            yield lambda sidx=sidx, ph=ph: kv_empty[sidx].ok(ph ^ 1)
            copies.append((sidx, what))
            if what == ("V", pad_tile, 1):
                st["pad_issued"] = True

    def pad_warp():
        p0 = ld_v(pad_tile)
        yield lambda: st["pad_issued"]
        for pos in (p0, p0 + 1):
            sidx, ph = pos % nstage, (pos // nstage) & 1
            yield lambda sidx=sidx, ph=ph: kv_full[sidx].ok(ph)
            if st["stage"][sidx] != ("V", pad_tile, pos - p0):
                errors.append(f"padding warp zeroes stage {sidx} holding {st['stage'][sidx]}")
        st["zeroed"] = pad_tile
        v_clean.arrive()

    def mma():
        yield lambda: q_full.ok(0)

        def issue_qk(j):
            for h in (0, 1):
                pos = ld_k(j) + h
                sidx, ph = pos % nstage, (pos // nstage) & 1
                yield lambda sidx=sidx, ph=ph: kv_full[sidx].ok(ph)
                queue.extend([("qk", j, h, sidx, ("S", j & 1)), ("commit", kv_empty[sidx])])
            queue.append(("commit", s_full[j & 1]))

        for j in range(n_lead):
            yield from issue_qk(j)
        for j in range(n_tiles):
            yield lambda j=j: p_ready[j & 1].ok((j >> 1) & 1)
            if j == pad_tile:
                yield lambda: v_clean.ok(0)
            for h in (0, 1):
                pos = ld_v(j) + h
                sidx, ph = pos % nstage, (pos // nstage) & 1
                yield lambda sidx=sidx, ph=ph: kv_full[sidx].ok(ph)
                queue.extend([("pv", j, h, sidx, ("O", h)), ("commit", kv_empty[sidx])])
            queue.append(("commit", pv_done))
            if j + 2 < n_tiles:
                yield lambda j=j: pv_done.ok(j & 1)
                yield from issue_qk(j + 2)
        queue.append(("commit", drain))

    def softmax():
        for j in range(n_tiles):
            yield lambda j=j: s_full[j & 1].ok((j >> 1) & 1)
            if st["S"][j & 1] != j:
                errors.append(f"softmax reads S_{j & 1} holding {st['S'][j & 1]} for tile {j}")
            if j > 0 and rng.random() < 0.5:   # the running max grew: rescale O
                yield lambda j=j: pv_done.ok((j - 1) & 1)
                if st["O"] != [j, j]:
                    errors.append(f"softmax rescales O holding {st['O']} tiles at tile {j}")
            st["P"][j & 1] = j
            st["S"][j & 1] = None   # P is written over S
            p_ready[j & 1].arrive()
        if n_tiles:
            if epilogue == "drain":
                yield lambda: drain.ok(0)
            else:
                yield lambda: pv_done.ok((n_tiles - 1) & 1)
            if st["O"] != [n_tiles, n_tiles]:
                errors.append(f"epilogue reads O holding {st['O']} of {n_tiles} tiles")

    partial_s = {}

    def execute():
        op = take_tensor_op(queue, rng)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, j, h, sidx, _ = op
        if st["stage"][sidx] != (("K" if kind == "qk" else "V"), j, h):
            errors.append(f"{kind} of tile {j} half {h} reads stage {sidx} holding {st['stage'][sidx]}")
        if kind == "qk":
            b = j & 1
            if not st["Q"]:
                errors.append(f"S of tile {j} reads Q before it landed")
            if st["P"][b] is not None and min(st["O"]) <= st["P"][b]:
                errors.append(f"S of tile {j} overwrites P of tile {st['P'][b]} before O += P V read it")
            if h == 0:
                partial_s[b] = j
            elif partial_s.get(b) == j:
                st["S"][b] = j
                st["P"][b] = None
        else:
            if j == pad_tile and st["zeroed"] != j:
                errors.append(f"P V of tile {j} reads V before its padding rows were zeroed")
            if st["P"][j & 1] != j or st["O"][h] != j:
                errors.append(f"O_{h} += P V of tile {j} reads P {st['P'][j & 1]} onto O of {st['O'][h]} tiles")
            st["O"][h] = j + 1

    roles = {"producer": producer(), "mma": mma(), "softmax": softmax()}
    if pad_tile is not None:
        roles["pad"] = pad_warp()
    waits = {}
    for name in list(roles):
        try:
            waits[name] = next(roles[name])
        except StopIteration:
            del roles[name]
    while roles or queue or copies:
        moves = [("role", r) for r in roles if waits[r]()]
        if queue:
            moves.append(("tensor", None))
        moves += [("copy", i) for i in range(len(copies))]
        if not moves:
            return [f"deadlock: {sorted(roles)} waiting"]
        kind, x = rng.choice(moves)
        if kind == "role":
            try:
                waits[x] = roles[x].send(None)
            except StopIteration:
                del roles[x]
        elif kind == "tensor":
            execute()
        else:
            sidx, what = copies.pop(x)
            if sidx == "Q":
                st["Q"] = True
                q_full.arrive()
            else:
                st["stage"][sidx] = what
                kv_full[sidx].arrive()
        if errors:
            return errors
    return errors


@pytest.mark.parametrize("nstage", [2, 4, 5, 7])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 17])
def test_wide_pipeline_is_clean(n, nstage):
    for trial in range(150):
        assert run_wide(n, nstage, trial) == [], f"n {n}, nstage {nstage}, seed {trial}"


@pytest.mark.parametrize("n", [1, 4, 16])
def test_wide_padding_warp_zeroes_the_right_tile(n):
    for trial in range(80):
        for pad in sorted({0, n // 2, n - 1}):
            assert run_wide(n, 5, trial, pad_tile=pad) == [], f"n {n}, pad {pad}, seed {trial}"


def test_wide_parity_epilogue_can_read_o_early():
    # with two score buffers the product of tile n - 2 may still be pending
    # when P_{n-1} is stored, so a parity wait for the last product can pass
    # on the completion of tile n - 3: the drain barrier is needed
    bad = sum(bool(run_wide(n, 5, trial, epilogue="parity")) for n in (5, 8, 17) for trial in range(300))
    assert bad > 0


def run_chain(units, nstage, seed, pad=None, q_handoff="count", o_free_wait=True, q_free_wait=True):
    """One random interleaving of the unit-chaining kernel (attn_chain): one
    CTA walks a list of work units (tile counts; 0 = a unit with nothing to
    attend, whose rows are written as zeros without any hand-off).  Units with
    tiles are numbered kappa = 0, 1, ...; their key tiles form one stream J.
    The per-tile protocol is the one-tile kernel's: two MMA threads, scores
    three tiles ahead into S[J % 2], a single P buffer written once the
    previous P V has completed.  At unit changes:
      Q: the unit warps copy Q_kappa from a single shared-memory buffer
        into the single tensor-memory Q buffer once the softmax has seen the
        last score tile of unit kappa - 1 (its Q K^T are then complete), send
        o of unit kappa - 1 out through the shared buffer, then load
        Q_{kappa+1} into it themselves (the producer,
        which runs three tiles ahead over several short units, would have to
        wait for that copy before its next K load: a cycle through the
        epilogue, which waits for a P V whose V comes after that K), and
        count the copy into q_ready; an MMA thread waits for q_ready > kappa
        before its first Q K^T of unit kappa (q_handoff="parity": a phase
        wait instead);
      O: the MMA thread of a unit's last tile commits o_full after its P V;
        the unit warps read O and the row sums (two slots) and free O; the
        first P V of the next unit (no accumulate) waits for that.
    pad: stream tiles whose V rows a padding warp zeroes (issued count, then
    the stage's phase) before their P V.  o_free_wait / q_free_wait=False
    drop those waits (planted mistakes).  Returns the list of violations."""
    rng = random.Random(seed)
    tiles, kap = [], []  # stream tile -> (unit, j, kappa); unit -> kappa or None
    kappa = 0
    for u, n in enumerate(units):
        kap.append(kappa if n else None)
        tiles.extend((u, j, kappa) for j in range(n))
        kappa += bool(n)
    N = len(tiles)
    pad = set(pad or ())
    pad_order = sorted(pad)
    kv_full = [Bar() for _ in range(nstage)]
    kv_empty = [Bar() for _ in range(nstage)]
    s_full, s_read = [Bar(), Bar()], [Bar(), Bar()]
    p_ready, pv_done = [Bar(), Bar()], [Bar(), Bar()]
    q_sfull, q_free, q_full = Bar(), Bar(), Bar()
    o_full, o_free = Bar(), Bar()
    l_full, l_free = [Bar(), Bar()], [Bar(), Bar()]
    st = {"Qs": None, "Qt": None, "q_ready": 0, "S": [None, None], "P": None, "O": None, "O_read": True,
          "l": [None, None], "stage": [None] * nstage, "v_issued": 0, "cleaned": 0, "zeroed": set()}
    queues = {0: [], 1: []}
    copies, errors = [], []

    def ld_v(J):
        return min(J + 4, N) + J

    def ld_k(J):
        return J if J < 3 else 2 * J - 3

    def bpar(J):
        return (J >> 1) & 1

    def producer():
        order = [("K", J) for J in range(min(3, N))]
        for J in range(N):
            if J + 3 < N:
                order.append(("K", J + 3))
            order.append(("V", J))
        for pos, (kind, J) in enumerate(order):
            assert pos == (ld_k(J) if kind == "K" else ld_v(J))
            sidx, ph = pos % nstage, (pos // nstage) & 1
            yield lambda sidx=sidx, ph=ph: kv_empty[sidx].ok(ph ^ 1)
            copies.append((sidx, (kind, J)))
            if kind == "V":
                st["v_issued"] = J + 1

    def pad_warp():
        for i, J in enumerate(pad_order):
            pos = ld_v(J)
            sidx, ph = pos % nstage, (pos // nstage) & 1
            yield lambda J=J: st["v_issued"] > J
            yield lambda sidx=sidx, ph=ph: kv_full[sidx].ok(ph)
            if st["stage"][sidx] != ("V", J):
                errors.append(f"padding warp zeroes stage {sidx} holding {st['stage'][sidx]}, not V_{J}")
            st["zeroed"].add(J)
            st["cleaned"] = i + 1

    def mma(p):
        if N <= p:
            return
        seen = [-1]

        def issue_qk(J):
            k = tiles[J][2]
            if k != seen[0]:
                if q_handoff == "count":
                    yield lambda k=k: st["q_ready"] > k
                else:
                    yield lambda k=k: q_full.ok(k & 1)
                seen[0] = k
            pos = ld_k(J)
            sidx, ph = pos % nstage, (pos // nstage) & 1
            yield lambda sidx=sidx, ph=ph: kv_full[sidx].ok(ph)
            if J >= 2:
                yield lambda J=J: s_read[J & 1].ok(bpar(J - 2))
            queues[p].extend([("qk", J, sidx, ("S", J & 1)), ("commit", s_full[J & 1]), ("commit", kv_empty[sidx])])

        yield from issue_qk(p)
        if p == 1 and N > 2:
            yield from issue_qk(2)
        for J in range(p, N, 2):
            u, j, k = tiles[J]
            pos = ld_v(J)
            sidx, ph = pos % nstage, (pos // nstage) & 1
            yield lambda sidx=sidx, ph=ph: kv_full[sidx].ok(ph)
            yield lambda J=J: p_ready[J & 1].ok(bpar(J))
            if j == 0 and k >= 1 and o_free_wait:
                yield lambda k=k: o_free.ok((k - 1) & 1)
            if J in pad:
                idx = pad_order.index(J)
                yield lambda idx=idx: st["cleaned"] > idx
            queues[p].extend([("pv", J, sidx, ("O",)), ("commit", pv_done[p]), ("commit", kv_empty[sidx])])
            if j == units[u] - 1:
                queues[p].append(("commit", o_full))
            if J + 3 < N:
                yield from issue_qk(J + 3)

    def softmax():
        J = 0
        for u, n in enumerate(units):
            if not n:
                continue
            k = kap[u]
            for j in range(n):
                yield lambda J=J: s_full[J & 1].ok(bpar(J))
                if st["S"][J & 1] != J:
                    errors.append(f"softmax reads S_{J & 1} holding {st['S'][J & 1]} for tile {J}")
                if j == n - 1:
                    q_free.arrive()  # every Q K^T of the unit has completed
                if j > 0 and rng.random() < 0.4:  # the running max grew: rescale O
                    yield lambda J=J: pv_done[(J - 1) & 1].ok(bpar(J - 1))
                    if st["O"] != (u, j):
                        errors.append(f"softmax rescales O holding {st['O']} at tile {j} of unit {u}")
                st["S"][J & 1] = ("read", J)
                s_read[J & 1].arrive()
                if J > 0:
                    yield lambda J=J: pv_done[(J - 1) & 1].ok(bpar(J - 1))
                st["P"] = J
                p_ready[J & 1].arrive()
                J += 1
            yield lambda k=k: l_free[k & 1].ok(((k >> 1) & 1) ^ 1)
            st["l"][k & 1] = u
            l_full[k & 1].arrive()

    def unit_warps():
        prev = None

        def epilogue(u, k, n):
            yield lambda k=k: o_full.ok(k & 1)
            yield lambda k=k: l_full[k & 1].ok((k >> 1) & 1)
            if st["O"] != (u, n):
                errors.append(f"epilogue of unit {u} reads O holding {st['O']}")
            if st["l"][k & 1] != u:
                errors.append(f"epilogue of unit {u} reads the row sums of unit {st['l'][k & 1]}")
            st["O_read"] = True
            l_free[k & 1].arrive()
            o_free.arrive()

        if N:
            copies.append(("Qs", 0))
        for u, n in enumerate(units):
            if not n:
                continue
            k = kap[u]
            if k >= 1 and q_free_wait:
                yield lambda k=k: q_free.ok((k - 1) & 1)
            yield lambda k=k: q_sfull.ok(k & 1)
            if st["Qs"] != k:
                errors.append(f"unit warps copy the shared Q buffer holding {st['Qs']} as Q of unit {k}")
            for p in (0, 1):
                for op in queues[p]:
                    if op[0] == "qk" and tiles[op[1]][2] != k:
                        errors.append(f"Q of unit {k} overwrites tensor memory before Q K^T of tile {op[1]}")
            st["Qt"] = k
            st["q_ready"] += 1
            q_full.arrive()
            if prev is not None:
                yield from epilogue(*prev)  # o of the previous unit goes out through the buffer
            if k + 1 < kappa:  # then the next unit's Q comes in through it
                copies.append(("Qs", k + 1))
            prev = (u, k, n)
        if prev is not None:
            yield from epilogue(*prev)

    def execute(p):
        op = take_tensor_op(queues[p], rng)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, J, sidx, acc = op
        u, j, k = tiles[J]
        if kind == "qk":
            if st["stage"][sidx] != ("K", J):
                errors.append(f"Q K^T of tile {J} reads stage {sidx} holding {st['stage'][sidx]}")
            if st["Qt"] != k:
                errors.append(f"Q K^T of tile {J} (unit {k}) reads the Q of unit {st['Qt']}")
            if isinstance(st["S"][J & 1], int):
                errors.append(f"Q K^T of tile {J} overwrites unread scores of tile {st['S'][J & 1]}")
            st["S"][J & 1] = J
        else:
            if st["stage"][sidx] != ("V", J):
                errors.append(f"P V of tile {J} reads stage {sidx} holding {st['stage'][sidx]}")
            if st["P"] != J:
                errors.append(f"P V of tile {J} reads P of tile {st['P']}")
            if J in pad and J not in st["zeroed"]:
                errors.append(f"P V of tile {J} reads V before its padding rows were zeroed")
            if j == 0:
                if not st["O_read"]:
                    errors.append(f"P V of tile {J} overwrites O before the epilogue read it")
                st["O"], st["O_read"] = (u, 1), False
            else:
                if st["O"] != (u, j):
                    errors.append(f"P V of tile {J} accumulates onto O holding {st['O']}")
                st["O"] = (u, j + 1)

    roles = {"producer": producer(), "mma0": mma(0), "mma1": mma(1), "softmax": softmax(),
             "units": unit_warps()}
    if pad:
        roles["pad"] = pad_warp()
    waits = {}
    for name in list(roles):
        try:
            waits[name] = next(roles[name])
        except StopIteration:
            del roles[name]
    while roles or queues[0] or queues[1] or copies:
        moves = [("role", r) for r in roles if waits[r]()]
        moves += [("tensor", p) for p in (0, 1) if queues[p]]
        moves += [("copy", i) for i in range(len(copies))]
        if not moves:
            return [f"deadlock: {sorted(roles)} waiting"]
        kind, x = rng.choice(moves)
        if kind == "role":
            try:
                waits[x] = roles[x].send(None)
            except StopIteration:
                del roles[x]
        elif kind == "tensor":
            execute(x)
        else:
            dst, what = copies.pop(x)
            if dst == "Qs":
                st["Qs"] = what
                q_sfull.arrive()
            else:
                st["stage"][dst] = what
                kv_full[dst].arrive()
        if errors:
            return errors
    return errors


def _chain_units(rng):
    return [rng.choice([0, 1, 1, 2, 3, 4, 4, 6]) for _ in range(rng.randint(1, 8))]


@pytest.mark.parametrize("nstage", [4, 6, 7])
def test_chain_pipeline_is_clean(nstage):
    rng = random.Random(100 + nstage)
    for trial in range(400):
        units = _chain_units(rng)
        assert run_chain(units, nstage, trial) == [], f"units {units}, seed {trial}"


def test_chain_padding_tiles():
    rng = random.Random(5)
    for trial in range(300):
        units = _chain_units(rng)
        n = sum(units)
        pad = sorted(rng.sample(range(n), min(n, 3))) if n else []
        assert run_chain(units, 6, trial, pad=pad) == [], f"units {units}, pad {pad}, seed {trial}"


def test_chain_parity_handoff_of_q_can_alias():
    # an MMA thread may issue no score product of a one-tile unit, and then a
    # phase wait no longer tells unit k's Q from unit k - 2's
    rng = random.Random(11)
    bad = sum(bool(run_chain(_chain_units(rng), 6, trial, q_handoff="parity")) for trial in range(1500))
    assert bad > 0


def test_chain_without_the_o_free_wait_overwrites_o():
    bad = sum(bool(run_chain([3, 2, 4, 1, 3], 6, trial, o_free_wait=False)) for trial in range(300))
    assert bad > 0


def test_chain_without_the_q_free_wait_overwrites_q():
    bad = sum(bool(run_chain([3, 2, 4, 1, 3], 6, trial, q_free_wait=False)) for trial in range(300))
    assert bad > 0
