"""A host-side model of the streaming kernel's slot-ring protocol.

Agents per CTA: one producer (issues bulk copies into a ring of NS slots),
one fold warp, W consumer warps; C CTAs per cluster exchange tile partials.
mbarriers follow the PTX rules: a phase completes when its pending arrival
count reaches zero and its expected bytes have landed; a parity wait succeeds
when the given parity is that of the phase before the current one (so a wait
two phases ahead succeeds wrongly).  The model drives every agent with random
speeds and random copy latencies and asserts that each read of a slot sees
the item it expects and that nothing deadlocks.

It mirrors the kernel's waits: full/empty per slot, rowdone/lseready/
partfree/xbar per row buffer, and the per-slot issued-item number (`seq`)
that consumers wait for before the full-barrier parity.

The exchange between the C CTAs of a cluster is asynchronous.  Row n is
folded by one CTA, the folder F(n) = n mod C: every other CTA sends it its
shard of partials and its target-logit record with remote stores that
complete on the folder's xbar barrier after a random delay; the folder folds
and sends the LSE back to every peer, completing on their lsebar barriers.
Every CTA arrives once per row on xbar and lsebar (with expect-tx where it
receives), so both barriers have one phase per row.  A CTA releases a row's
buffers (partfree) only once it holds the row's LSE.  The fold warp is an
event loop that pushes, folds and releases rows as each becomes possible.
The folder reads the partials over several steps and checks that nothing
overwrote them.
"""
import random


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0
        self.tx = 0

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise ProtocolError("more arrivals than the phase expects")
        self.check()

    def check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def try_wait(self, par):
        return par != (self.phase & 1)


class ProtocolError(AssertionError):
    pass


def block_schedule(mode, rows, skew=1):
    """Blocks of nch items the producer issues, in order: ('A' | 'B', row)."""
    if mode == "fwd":
        return [("A", n) for n in range(rows)]
    if mode == "bwd":
        return [("B", n) for n in range(rows)]
    if mode == "fused":
        return [("A", n) for n in range(rows)]  # one load per row; phase B reuses the resident slots
    # fused_l2 with skew S: A(0..S-1), then A(n+S), B(n) for each n
    seq = [("A", n) for n in range(min(skew, rows))]
    for n in range(rows):
        if n + skew < rows:
            seq.append(("A", n + skew))
        seq.append(("B", n))
    return seq


def row_skip_safe(W, ntl, span, first_lim):
    """The planner's condition for skipping rows without a tile (row_skip_safe in logp_stream.cu):
    every warp's first row below first_lim and its consecutive rows at most span apart.  The
    forward takes span = rbufs, first_lim = 2*rbufs; the L2 fused schedule span = rbufs - skew,
    first_lim = rbufs."""
    if ntl >= W:
        return False
    step = ntl % W
    for w in range(W):
        last, r = -1, 0
        for n in range(2 * W + 2 * first_lim):
            if (w - r) % W < ntl:
                if (n >= first_lim) if last < 0 else (n - last > span):
                    return False
                last = n
            r = (r + step) % W
        if last < 0:
            return False
    return True


def skip_condition(mode, W, ntl, rbufs, skew):
    """row_skip_safe with the mode's span and first-row limit (False for modes that never skip)."""
    if mode == "fwd":
        return row_skip_safe(W, ntl, rbufs, 2 * rbufs)
    if mode == "fused_l2":
        return rbufs > skew and row_skip_safe(W, ntl, rbufs - skew, rbufs)
    return False


def simulate(mode, rows, C, NT, tps, NS, W, seed=0, seqcheck=True, max_delay=80, rbufs=2, skew=1,
             producers=1, producer_seqcheck=True, row_skip=None, speeds=(0.02, 0.1, 0.5, 1.0)):
    """mode: 'fwd' | 'bwd' | 'fused' | 'fused_l2'; rbufs row buffers, fused_l2 row skew;
    producers: producer warps per CTA, producer p issuing the items i with i mod producers == p
    (each waits until the slot's previous item is issued before its empty-barrier parity,
    unless producer_seqcheck is off).

    row_skip: warps skip the rows in which they have no tile (the forward and the L2 fused
    schedule; None: the planner's condition).

    speeds: the chances per step that an agent moves, one drawn per agent (a very slow agent
    stands for a warp held up for a long time).

    Raises ProtocolError on a stale read or a deadlock."""
    rng = random.Random(seed)
    ntl = NT // C
    S = skew if mode == "fused_l2" else 1
    if row_skip is None:
        row_skip = skip_condition(mode, W, ntl, rbufs, S)
    nch = (ntl + tps - 1) // tps
    R = rbufs
    pushes = []  # in flight: [delay, receiver CTA, kind, buffer, index, value]

    def folder(n):
        return n % C

    class CTA:
        pass

    ctas = []
    for r in range(C):
        c = CTA()
        c.rank = r
        c.full = [Bar(1) for _ in range(NS)]
        c.empty = [Bar(tps) for _ in range(NS)]
        c.hdr = [None] * NS
        c.seq = [None] * NS
        c.data = [None] * NS
        c.inflight = []
        c.rowdone = [Bar(min(W, ntl) if row_skip else W) for _ in range(R)]
        c.lseready = [Bar(1) for _ in range(R)]
        c.partfree = [Bar(1) for _ in range(R)]
        c.xbar = [Bar(1) for _ in range(R)]
        c.lsebar = [Bar(1) for _ in range(R)]
        c.xt = [[None] * C for _ in range(R)]
        c.part = [[None] * NT for _ in range(R)]
        c.lse = [None] * R
        c.xtrow = [None] * R
        ctas.append(c)

    def ring(i):
        return i % NS, (i // NS) & 1

    def chunk_of(l):
        ch = l // tps
        kf = ch * tps
        kl = min(kf + tps, ntl)
        return ch, (1 + tps - (kl - kf)) if l == kl - 1 else 1

    def wait(bar, par):
        while not bar.try_wait(par):
            yield "wait"

    def wait_item(c, s, par, i):
        if seqcheck:
            while c.seq[s] != i:
                yield "wait"
        yield from wait(c.full[s], par)

    def check_slot(c, s, i, where):
        if c.hdr[s] != i or c.data[s] != i:
            raise ProtocolError(f"{mode} {where}: slot {s} holds item {c.hdr[s]}/{c.data[s]}, expected {i}")

    sched = block_schedule(mode, rows, S)
    block_index = {blk: b for b, blk in enumerate(sched)}

    def item_of(phase, n, ch):
        if mode == "fused":
            return n * nch + ch
        return block_index[(phase, n)] * nch + ch

    def producer(c, pid):
        i = 0
        for _ in sched:
            for _ in range(nch):
                if i % producers != pid:
                    i += 1
                    continue
                s, par = ring(i)
                if producer_seqcheck and i >= NS:
                    while c.seq[s] != i - NS:
                        yield "wait"
                yield from wait(c.empty[s], par ^ 1)
                if c.hdr[s] is not None and c.hdr[s] != i - NS:
                    raise ProtocolError(f"{mode} producer {pid} reused slot {s} for item {i} "
                                        f"while it held item {c.hdr[s]}")
                c.hdr[s] = i
                c.seq[s] = i
                c.data[s] = None
                c.full[s].tx += 1
                c.full[s].arrive()
                c.inflight.append([rng.randint(1, max_delay), s, i])
                i += 1
                yield "issue"

    def tiles_of(w, n):
        return range((w - n * ntl) % W, ntl, W)

    def phase_a(c, w, n):
        b = n % R
        if row_skip and not tiles_of(w, n):  # a warp without tiles skips the row
            return
        if n >= R:
            yield from wait(c.partfree[b], (n // R - 1) & 1)
        for l in tiles_of(w, n):
            ch, share = chunk_of(l)
            i = item_of("A", n, ch)
            s, par = ring(i)
            yield from wait_item(c, s, par, i)
            check_slot(c, s, i, "phase A")
            c.part[b][c.rank * ntl + l] = n
            c.xtrow[b] = n
            yield "tile"
            if mode in ("fwd", "fused_l2"):
                c.empty[s].arrive(share)
        c.rowdone[b].arrive()
        yield "arrived"

    def phase_b(c, w, n):
        if mode in ("fused", "fused_l2") and c.lse[n % R] != n:
            raise ProtocolError(f"{mode} phase B of row {n} read the LSE of row {c.lse[n % R]}")
        for l in tiles_of(w, n):
            ch, share = chunk_of(l)
            i = item_of("A" if mode == "fused" else "B", n, ch)
            s, par = ring(i)
            if mode in ("bwd", "fused_l2"):
                yield from wait_item(c, s, par, i)
            check_slot(c, s, i, "phase B")
            yield "grad"
            c.empty[s].arrive(share)

    def consumer(c, w):
        if mode == "bwd":
            for n in range(rows):
                yield from phase_b(c, w, n)
        elif mode == "fwd":
            for n in range(rows):
                yield from phase_a(c, w, n)
        else:
            for n in range(min(S, rows)):
                yield from phase_a(c, w, n)
            for n in range(rows):
                if n + S < rows:
                    yield from phase_a(c, w, n + S)
                if row_skip and not tiles_of(w, n):  # no tile: neither the LSE nor phase B
                    continue
                yield from wait(c.lseready[n % R], (n // R) & 1)
                yield from phase_b(c, w, n)

    def do_push(c, m):
        b = m % R
        if C > 1:
            f = ctas[folder(m)]
            if f is c:
                c.xbar[b].tx += (C - 1) * (ntl + 1)  # expect the peers' shards and records
                c.xbar[b].arrive()
                c.lsebar[b].arrive()
            else:
                c.xbar[b].arrive()
                c.lsebar[b].tx += 1  # expect the LSE
                c.lsebar[b].arrive()
                for k in range(c.rank * ntl, (c.rank + 1) * ntl):
                    pushes.append([rng.randint(1, max_delay), f, "part", b, k, c.part[b][k]])
                pushes.append([rng.randint(1, max_delay), f, "xt", b, c.rank, c.xtrow[b]])

    def fold(c):
        # The fold warp as an event loop: push rows in order as their phase A
        # completes, fold this CTA's rows as soon as their shards are in, and
        # release rows in order as their LSE is known.  No step waits for
        # another: a row's fold never waits for an earlier row's LSE.
        np_, nr = 0, 0
        nf = c.rank if C > 1 else 0
        step = C if C > 1 else 1
        while nr < rows:
            progressed = False
            if np_ < rows and c.rowdone[np_ % R].try_wait((np_ // R) & 1):
                do_push(c, np_)
                np_ += 1
                progressed = True
            if nf < rows and nf < np_ and (C == 1 or c.xbar[nf % R].try_wait((nf // R) & 1)):
                n, b = nf, nf % R
                if any(v != n for v in c.part[b]) or any(c.xt[b][j] != n for j in range(C) if C > 1 and j != c.rank):
                    raise ProtocolError(f"{mode} fold of row {n} saw partials of rows "
                                        f"{sorted(set(map(str, c.part[b])))}")
                yield "fold"
                yield "fold"
                if any(v != n for v in c.part[b]):
                    raise ProtocolError(f"{mode} partials of row {n} were overwritten during its fold")
                c.lse[b] = n
                for peer in ctas:
                    if peer is not c:
                        pushes.append([rng.randint(1, max_delay), peer, "lse", b, 0, n])
                nf += step
                progressed = True
            if nr < np_:
                b = nr % R
                ready = nr < nf if (C == 1 or folder(nr) == c.rank) else c.lsebar[b].try_wait((nr // R) & 1)
                if ready:
                    if c.lse[b] != nr:
                        raise ProtocolError(f"{mode} CTA {c.rank} released row {nr} holding the LSE of row {c.lse[b]}")
                    if mode in ("fused", "fused_l2"):
                        c.lseready[b].arrive()
                    c.partfree[b].arrive()
                    nr += 1
                    progressed = True
            yield "step" if progressed else "wait"

    agents = []
    for c in ctas:
        agents.extend(producer(c, pid) for pid in range(producers))
        if mode != "bwd":
            agents.append(fold(c))
        agents.extend(consumer(c, w) for w in range(W))
    speed = {id(a): rng.choice(list(speeds)) for a in agents}
    live = list(agents)
    idle = 0
    while live:
        progressed = False
        for f in pushes:
            f[0] -= 1
        for f in [f for f in pushes if f[0] <= 0]:
            pushes.remove(f)
            _, peer, kind, b, k, v = f
            if kind == "part":
                peer.part[b][k] = v
            elif kind == "xt":
                peer.xt[b][k] = v
            else:
                peer.lse[b] = v
            bar = peer.lsebar[b] if kind == "lse" else peer.xbar[b]
            bar.tx -= 1
            bar.check()
            progressed = True
        for c in ctas:
            for f in c.inflight:
                f[0] -= 1
            for f in [f for f in c.inflight if f[0] <= 0]:
                c.inflight.remove(f)
                c.data[f[1]] = f[2]
                c.full[f[1]].tx -= 1
                c.full[f[1]].check()
                progressed = True
        picked = [a for a in live if rng.random() < speed[id(a)]] or [rng.choice(live)]
        rng.shuffle(picked)
        for a in picked:
            try:
                if next(a) != "wait":
                    progressed = True
            except StopIteration:
                live.remove(a)
                progressed = True
        idle = 0 if progressed else idle + 1
        if idle > 5000:
            raise ProtocolError(f"{mode}: deadlock with {len(live)} agents waiting")
