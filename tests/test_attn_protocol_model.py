"""Model check of the persistent attention kernel's barrier protocol (attention.cu).

Roles, each in the program order of the kernel: the TMA producer, one MMA issuer per query tile
(tile 0 and tile 1 of a work item), and the softmax warps of each tile.  Asynchronous work is
modelled as such: a TMA copy lands on its "full" barrier at an arbitrary later time, and the
tensor-core operations of an issuer complete in that issuer's program order, each commit arriving
on its barrier only once everything the issuer issued before it has completed, at an arbitrary
later time.  Random interleavings of all of this must

* never deadlock,
* pass every parity wait exactly when the phase it means has completed (the barrier is never two
  phases ahead of the waiter, which a parity cannot tell apart),
* never overwrite a shared-memory tile (Q of a tile, K or V of a ring slot) while an issued product
  that reads it has not completed, and let every product read the block it is meant to,
* let the softmax write P_x into tensor memory only after the previous P_x V has completed, read
  O_x only after the item's last product into it, and let the next item overwrite O_x only after
  that read,
* write every query block of every (head, sequence) exactly once.

The model covers the work lists of the kernel (units of a heaviest and a lightest item) for small
head counts, sequence counts and grids."""
import random
from collections import deque

import pytest


def work(n_qblk, heads, nseq):
    n_pairs = (n_qblk + 1) >> 1
    upg = (n_pairs + 1) >> 1
    return n_pairs, upg, upg * heads * nseq


def items_of(cta, grid, n_qblk, heads, nseq):
    """The items CTA `cta` walks, in order (the kernel's AttnWork / attn_item / attn_unit_items)."""
    n_pairs, upg, units = work(n_qblk, heads, nseq)
    out = []
    for u in range(cta, units, grid):
        k = u % upg
        nit = 2 if k < n_pairs - 1 - k else 1
        for half in range(nit):
            g = u // upg
            ip = n_pairs - 1 - k if half == 0 else k
            q0 = 2 * ip
            nt = 2 if q0 + 1 < n_qblk else 1
            out.append(dict(hd=g % heads, sq=g // heads, q0=q0, ntiles=nt, nblk=q0 + nt))
    return out


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arr, self.done = name, count, 0, 0

    def arrive(self, n=1):
        self.arr += n
        assert self.arr <= self.count, f"{self.name}: more arrivals than the barrier counts"
        if self.arr == self.count:
            self.arr, self.done = 0, self.done + 1

    def passes(self, parity, intended):
        """A parity wait for the `intended`-th completion (1-based)."""
        by_parity = (self.done & 1) != parity
        by_count = self.done >= intended
        assert self.done <= intended, f"{self.name}: {self.done} completions, the waiter means #{intended}"
        assert by_parity == by_count, f"{self.name}: parity {parity} vs completion #{intended} ({self.done})"
        return by_count


class Model:
    # planted mistake for the test below: the producer waits only for the release of the last tile
    # that consumed a ring slot (right with one issuer, whose products complete in order; wrong with one
    # issuer per tile)
    last_consumer_only = False

    def __init__(self, its, n_qblk, rng):
        self.its, self.n_qblk, self.rng = its, n_qblk, rng
        self.bars = {}
        for x in range(2):
            for nm in ("QF", "QE", "SF", "PD"):
                self.bars[f"{nm}{x}"] = Bar(f"{nm}{x}", 1)
            for nm in ("PF", "OF"):
                self.bars[f"{nm}{x}"] = Bar(f"{nm}{x}", 4)
            for b in range(2):
                self.bars[f"KE{x}{b}"] = Bar(f"KE{x}{b}", 1)
                self.bars[f"VE{x}{b}"] = Bar(f"VE{x}{b}", 1)
        for b in range(2):
            self.bars[f"KF{b}"] = Bar(f"KF{b}", 1)
            self.bars[f"VF{b}"] = Bar(f"VF{b}", 1)
        for x in range(2):
            self.bars[f"TK{x}"] = Bar(f"TK{x}", 1)  # issuer x's turn
        self.tma = []                       # copies in flight: (buffer, content, full barrier)
        self.smem = {}                      # buffer -> content that has landed
        self.readers = {}                   # buffer -> products issued and not completed that read it
        self.pipe = [deque(), deque()]      # per issuer: ("mma", reads, writes) / ("commit", barrier)
        self.pv_pending = [0, 0]            # P_x V issued and not completed, per tile
        self.o_last_done = [0, 0]           # items whose last product into O_x has completed
        self.o_read = [0, 0]                # items whose O_x the softmax has read
        self.writes = {}
        self.order = []                     # (item, block or -1 for the first products, tile) as issued

    def wait(self, name, parity, intended):
        return self.bars[name].passes(parity, intended)

    # ---- asynchronous completions
    def land_copy(self):
        i = self.rng.randrange(len(self.tma))
        buf, content, bar = self.tma.pop(i)
        self.smem[buf] = content
        if not any(t[2] == bar for t in self.tma):  # the last copy of its phase has landed
            self.bars[bar].arrive()

    def complete_one(self, x):
        op = self.pipe[x].popleft()
        if op[0] == "mma":
            _, reads, kind, item = op
            for buf in reads:
                self.readers[buf] -= 1
            if kind == "pv":
                self.pv_pending[x] -= 1
            if kind == "pv_last":
                self.pv_pending[x] -= 1
                self.o_last_done[x] = max(self.o_last_done[x], item + 1)
        else:
            self.bars[op[1]].arrive()

    # ---- the tensor-core operations an issuer places in its pipe
    def mma(self, x, reads, expect, kind="qk", item=0):
        for buf, content in zip(reads, expect):
            assert self.smem.get(buf) == content, f"product of tile {x} reads {buf}={self.smem.get(buf)}, wants {content}"
            self.readers[buf] = self.readers.get(buf, 0) + 1
        if kind.startswith("pv"):
            self.pv_pending[x] += 1
        self.pipe[x].append(("mma", reads, kind, item))

    def commit(self, x, bar):
        self.pipe[x].append(("commit", bar))

    def copy(self, buf, content, bar):
        assert self.readers.get(buf, 0) == 0, f"copy into {buf} while a product still reads it"
        self.smem.pop(buf, None)
        self.tma.append((buf, content, bar))

    # ---- roles (generators that yield while a wait does not pass)
    def producer(self):
        gb = 0
        qst = 0    # bit x: parity of the items tile x took part in; bit x + 2: there was one
        cons = 0   # bit 2b + x: tile x consumes the block now in ring slot b
        upar = 0   # bit 2b + x: parity of the blocks of slot b that tile x consumed
        for ii, it in enumerate(self.its):
            for x in range(it["ntiles"]):
                if (qst >> (x + 2)) & 1:
                    nq = self.q_items(ii, x)
                    while not self.wait(f"QE{x}", ((qst >> x) & 1) ^ 1, nq):
                        yield
                self.copy(f"Q{x}", (ii, x), f"QF{x}")
                qst = (qst ^ (1 << x)) | (4 << x)
            for j in range(it["nblk"]):
                r = gb + j
                b = r & 1
                for x in self.releasing(cons, b):
                    n = self.slot_uses(b, x, r)
                    while not self.wait(f"KE{x}{b}", ((upar >> (2 * b + x)) & 1) ^ 1, n):
                        yield
                self.copy(f"K{b}", r, f"KF{b}")
                for x in self.releasing(cons, b):
                    n = self.slot_uses(b, x, r)
                    while not self.wait(f"VE{x}{b}", ((upar >> (2 * b + x)) & 1) ^ 1, n):
                        yield
                self.copy(f"V{b}", r, f"VF{b}")
                users = (1 if j <= it["q0"] else 0) | (2 if it["ntiles"] == 2 else 0)
                cons = (cons & ~(3 << (2 * b))) | (users << (2 * b))
                upar ^= users << (2 * b)
            gb += it["nblk"]

    def releasing(self, cons, b):
        """The tiles whose release of ring slot b the producer waits for before refilling it."""
        users = [x for x in range(2) if (cons >> (2 * b + x)) & 1]
        return users[-1:] if self.last_consumer_only else users

    def q_items(self, upto, x):
        """Items before `upto` in which tile x took part (completions of QE_x the producer needs)."""
        return sum(1 for it in self.its[:upto] if x < it["ntiles"])

    def slot_uses(self, b, x, r):
        """Blocks of ring slot b before ring position r that tile x consumed."""
        n, gb = 0, 0
        for it in self.its:
            for j in range(it["nblk"]):
                rr = gb + j
                if rr >= r:
                    return n
                if rr & 1 == b and (x == 1 and it["ntiles"] == 2 or x == 0 and j <= it["q0"]):
                    n += 1
            gb += it["nblk"]
        return n

    def issuer(self, x):
        """Issuer of tile x.  The two issuers take turns (token barriers TK0, TK1) in the order one
        issuer would use: per block, tile 0's products, then tile 1's.  Each waits for its data first,
        then for its turn, issues its products, hands the turn over and only then commits."""
        gb = 0
        st = 0      # bit 0: item parity, bit 1: took part before, bit 2: P_FULL parity
        nitems = 0
        npf = 0
        ntok = 0    # turns received
        prev_nt = 0
        for ii, it in enumerate(self.its):
            q0, nblk, nt = it["q0"], it["nblk"], it["ntiles"]
            if x >= nt:
                gb += nblk
                prev_nt = nt
                continue
            qlast = q0 + x

            def turn(wait_turn):
                nonlocal ntok
                if wait_turn:
                    while not self.wait(f"TK{x}", ntok & 1, ntok + 1):
                        yield
                    ntok += 1

            # the item's first product S_x = Q_x K_0^T
            while not self.wait(f"QF{x}", st & 1, nitems + 1):
                yield
            while not self.wait(f"KF{gb & 1}", (gb >> 1) & 1, gb // 2 + 1):
                yield
            yield from turn(prev_nt == 2 if x == 0 else True)
            self.order.append((ii, -1, x))
            self.mma(x, [f"Q{x}", f"K{gb & 1}"], [(ii, x), gb])
            if nt == 2:
                self.bars[f"TK{1 - x}"].arrive()
            self.commit(x, f"SF{x}")
            self.commit(x, f"KE{x}{gb & 1}")
            if qlast == 0:
                self.commit(x, f"QE{x}")
            for j in range(qlast + 1):
                r, r1 = gb + j, gb + j + 1
                while not self.wait(f"VF{r & 1}", (r >> 1) & 1, r // 2 + 1):
                    yield
                if j < qlast:
                    while not self.wait(f"KF{r1 & 1}", (r1 >> 1) & 1, r1 // 2 + 1):
                        yield
                if j == 0 and (st >> 1) & 1:
                    while not self.wait(f"OF{x}", (st & 1) ^ 1, nitems):
                        yield
                    assert self.o_read[x] >= nitems, "O_x overwritten before the softmax read it"
                # tile 0 always waits for its turn in a two-tile item; tile 1 except after its own
                # product of block q0
                yield from turn(nt == 2 and (x == 0 or j <= q0))
                while not self.wait(f"PF{x}", (st >> 2) & 1, npf + 1):
                    yield
                self.order.append((ii, j, x))
                self.mma(x, [f"V{r & 1}"], [r], "pv_last" if j == qlast else "pv", nitems)
                if j < qlast:
                    self.mma(x, [f"Q{x}", f"K{r1 & 1}"], [(ii, x), r1])
                # hand over: tile 0 in a two-tile item; tile 1 unless its own product of block
                # q0 + 1 comes next
                if nt == 2 and (x == 0 or j != q0):
                    self.bars[f"TK{1 - x}"].arrive()
                self.commit(x, f"PD{x}")
                self.commit(x, f"VE{x}{r & 1}")
                st ^= 4
                npf += 1
                if j < qlast:
                    self.commit(x, f"SF{x}")
                    self.commit(x, f"KE{x}{r1 & 1}")
                    if j + 1 == qlast:
                        self.commit(x, f"QE{x}")
            st = (st ^ 1) | 2
            nitems += 1
            gb += nblk
            prev_nt = nt

    def softmax(self, x):
        cb = 0
        nitems = 0
        for it in self.its:
            if x >= it["ntiles"]:
                continue
            qblk = it["q0"] + x
            for j in range(qblk + 1):
                while not self.wait(f"SF{x}", cb & 1, cb + 1):
                    yield
                # no wait for the previous P_x V: S_FULL is committed after it by the same issuer
                assert self.pv_pending[x] == 0, "P_x written while a P_x V product is in flight"
                self.bars[f"PF{x}"].arrive(4)
                cb += 1
            while not self.wait(f"PD{x}", (cb - 1) & 1, cb):
                yield
            assert self.o_last_done[x] >= nitems + 1, "O_x read before its last product completed"
            self.o_read[x] = nitems + 1
            self.bars[f"OF{x}"].arrive(4)
            key = (it["hd"], it["sq"], qblk)
            if qblk < self.n_qblk:
                self.writes[key] = self.writes.get(key, 0) + 1
            nitems += 1

    def signature(self):
        return (tuple(b.done * 8 + b.arr for b in self.bars.values()), len(self.tma), len(self.pipe[0]),
                len(self.pipe[1]))

    def run(self):
        roles = [self.producer(), self.issuer(0), self.issuer(1), self.softmax(0), self.softmax(1)]
        alive = [True] * len(roles)
        stuck = 0
        while True:
            moves = [("role", i) for i in range(len(roles)) if alive[i]]
            moves += [("copy", 0)] * (1 if self.tma else 0)
            moves += [("pipe", x) for x in range(2) if self.pipe[x]]
            if not moves:
                break
            kind, i = self.rng.choice(moves)
            before = self.signature()
            if kind == "copy":
                self.land_copy()
            elif kind == "pipe":
                self.complete_one(i)
            else:
                try:
                    next(roles[i])
                except StopIteration:
                    alive[i] = False
            stuck = stuck + 1 if self.signature() == before else 0
            assert stuck < 2000, "deadlock: no role can move"
        assert all(v == 0 for v in self.readers.values())
        # the products went out in one issuer's order: per item the first products of tile 0 and 1,
        # then per key block tile 0's, then tile 1's
        want = []
        for ii, it in enumerate(self.its):
            want += [(ii, -1, x) for x in range(it["ntiles"])]
            want += [(ii, j, x) for j in range(it["nblk"]) for x in range(it["ntiles"]) if j <= it["q0"] + x]
        assert self.order == want


CASES = [(n_qblk, heads, nseq) for n_qblk in (1, 2, 3, 4, 5, 7, 8, 16) for heads, nseq in ((1, 1), (2, 1), (3, 2))]


@pytest.mark.parametrize("n_qblk,heads,nseq", CASES)
def test_attention_protocol(n_qblk, heads, nseq):
    n_pairs, upg, units = work(n_qblk, heads, nseq)
    rng = random.Random(n_qblk * 1000 + heads * 10 + nseq)
    writes = {}
    for grid in sorted({1, 2, 3, units}):
        if grid > units:
            continue
        writes = {}
        for cta in range(grid):
            for trial in range(3):
                m = Model(items_of(cta, grid, n_qblk, heads, nseq), n_qblk, rng)
                m.run()
            for k, v in m.writes.items():
                writes[k] = writes.get(k, 0) + v
        expect = {(h, s, q) for h in range(heads) for s in range(nseq) for q in range(n_qblk)}
        assert set(writes) == expect
        assert all(v == 1 for v in writes.values())


def test_model_catches_a_missing_wait():
    """The model is not vacuous: an issuer that skips its wait for the P hand-off is caught."""
    its = items_of(0, 1, 4, 1, 1)

    class Broken(Model):
        def wait(self, name, parity, intended):
            if name.startswith("PF"):
                return True
            return super().wait(name, parity, intended)

    failed = 0
    for seed in range(20):
        try:
            Broken(its, 4, random.Random(seed)).run()
        except AssertionError:
            failed += 1
    assert failed > 0


def test_model_catches_release_by_the_last_tile_only():
    """With one issuer per tile, a slot released by its last consumer alone may still be read by the
    other tile's products when it is refilled: the model must catch it."""
    its = items_of(0, 1, 8, 1, 1)

    class Broken(Model):
        last_consumer_only = True

    failed = 0
    for seed in range(30):
        try:
            Broken(its, 8, random.Random(seed)).run()
        except AssertionError as e:
            failed += 1
            assert "reads" in str(e) or "completions" in str(e), e  # a refill under a reader
    assert failed > 0
