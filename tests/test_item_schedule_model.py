"""A model of the per-item forward kernel's barrier protocol (no GPU).

The per-item blocks walk several rows ("items") with ring positions and
buffer counts that continue across rows, two or one Q buffers, and an O
hand-off barrier.  Every wait in the kernel is a parity wait on an mbarrier:
waiting for completion number k passes once the barrier has completed k + 1
times, and would miss its phase if the barrier could complete k + 2 times
before the waiter looks.  This model runs the kernel's three roles (producer,
MMA issuer, softmax warps) and its two asynchronous agents (the copy engine,
which completes tile and Q loads out of order, and the tensor pipe, which
runs MMA groups and commits in issue order) as interleaved processes over
barrier completion counts, with randomised scheduling, row lengths and
rescale decisions, and checks that
  * no run deadlocks,
  * no barrier ever completes a second time past a waiter's target, and
  * no wait is issued while its barrier still lacks the completion before
    the one it waits for
(together: the parity of every wait is unambiguous).
The waits, arrivals and commits follow k_bsa_forward_items in the order the
kernel issues them; the ring size S and the Q buffer count take the values of
the kernel's instantiations.
"""
import random

import pytest

KSBUF = 3


def ring_pos_k(j):
    return j if j < KSBUF else 2 * j - 2


def ring_pos_v(i, n):
    lead = min(n, KSBUF)
    mid = (i if i < n - KSBUF else n - KSBUF) if n - KSBUF > 0 else 0
    return lead + i + mid


def tile_is_v(t, n):
    lead = min(n, KSBUF)
    inter = 2 * (n - lead)
    return t >= lead and (t - lead >= inter or ((t - lead) & 1) == 0)


class Model:
    def __init__(self, rows, S, kqb, rng, producers=1):
        self.rows, self.S, self.kqb, self.rng = rows, S, kqb, rng
        self.count = {}          # barrier -> completions so far
        self.waiting = {}        # process name -> (barrier, target completion index)
        self.copies = []         # pending copy-engine completions (barrier names)
        self.pipe = []           # tensor pipe: in-order list of barrier names to complete
        if producers == 1:
            self.procs = {"producer": self.producer()}
        else:
            # the single-row kernel's gathered K/V: producer warps g take
            # tiles t with t % producers == g (one row, Q loaded once)
            assert len(rows) == 1
            self.procs = {f"producer{g}": self.gather_producer(g, producers) for g in range(producers)}
        self.procs.update({"mma": self.mma(), "softmax": self.softmax()})

    # a wait for completion number k passes when count > k; the model yields
    # the wait to the scheduler until then
    def wait(self, bar, k):
        return ("wait", bar, k)

    def complete(self, bar):
        c = self.count.get(bar, 0) + 1
        self.count[bar] = c
        for name, (b, k) in self.waiting.items():
            assert not (b == bar and c >= k + 2), f"{name} waiting for completion {k} of {bar}, now {c}"

    def producer(self):
        pos = 0
        qi = 0
        for n in self.rows:
            if n == 0:
                continue
            qb = qi % self.kqb
            if qi >= self.kqb:
                yield self.wait(("q_empty", qb), qi // self.kqb - 1)
            self.copies.append(("q_full", qb))
            for t in range(2 * n):
                slot = pos % self.S
                if pos >= self.S:
                    yield self.wait(("empty", slot), pos // self.S - 1)
                self.copies.append(("full", slot))
                pos += 1
            qi += 1

    def gather_producer(self, g, producers):
        n = self.rows[0]
        if g == 0 and n > 0:
            self.copies.append(("q_full", 0))
        for pos in range(g, 2 * n, producers):
            slot = pos % self.S
            if pos >= self.S:
                yield self.wait(("empty", slot), pos // self.S - 1)
            self.copies.append(("full", slot))  # the tile's 32 lane arrivals, once all copies landed

    def mma(self):
        pos = 0
        qi = 0
        g = 0
        for n in self.rows:
            if n == 0:
                continue
            qb = qi % self.kqb
            yield self.wait(("q_full", qb), qi // self.kqb)

            def issue_qk(j):
                nonlocal pos
                slot = pos % self.S
                yield self.wait(("full", slot), pos // self.S)
                self.pipe.append(("empty", slot))  # commit after QK_j (signals S_j)
                if self.kqb == 1 and j == n - 1:
                    self.pipe.append(("q_empty", 0))
                pos += 1

            for j in range(min(n, KSBUF)):
                yield from issue_qk(j)
            for i in range(n):
                gb = g + i
                yield self.wait(("p_full", gb % KSBUF), gb // KSBUF)
                if i == 0 and qi > 0:
                    yield self.wait(("o_free",), qi - 1)
                slot = pos % self.S
                yield self.wait(("full", slot), pos // self.S)
                self.pipe.append(("empty", slot))  # commit after PV_i
                pos += 1
                if i + KSBUF < n:
                    yield from issue_qk(i + KSBUF)
            if self.kqb == 2:
                self.pipe.append(("q_empty", qb))
            g += n
            qi += 1

    def softmax(self):
        t_glob = 0
        g = 0
        for n in self.rows:
            if n == 0:
                continue
            for j in range(n):
                pk = t_glob + ring_pos_k(j)
                yield self.wait(("empty", pk % self.S), pk // self.S)
                if j > 0 and self.rng.random() < 0.3:  # a rescale waits for PV_{j-1}
                    pv = t_glob + ring_pos_v(j - 1, n)
                    yield self.wait(("empty", pv % self.S), pv // self.S)
                self.complete(("p_full", (g + j) % KSBUF))
            pv = t_glob + ring_pos_v(n - 1, n)
            yield self.wait(("empty", pv % self.S), pv // self.S)
            self.complete(("o_free",))
            t_glob += 2 * n
            g += n

    def run(self, max_steps=200000):
        pending = dict.fromkeys(self.procs)
        state = {name: None for name in self.procs}
        for _ in range(max_steps):
            ready = []
            for name in list(pending):
                w = state[name]
                if w is None or self.count.get(w[1], 0) > w[2]:
                    ready.append(name)
            agents = (["copy"] if self.copies else []) + (["pipe"] if self.pipe else [])
            choices = ready + agents
            if not choices:
                assert not pending, f"deadlock: {[(n, state[n]) for n in pending]}"
                return
            c = self.rng.choice(choices)
            if c == "copy":
                self.complete(self.copies.pop(self.rng.randrange(len(self.copies))))
            elif c == "pipe":
                self.complete(self.pipe.pop(0))
            else:
                self.waiting.pop(c, None)
                try:
                    w = next(self.procs[c])
                    # a parity wait for completion k issued while the barrier
                    # has completed only k - 1 times would pass at once
                    assert self.count.get(w[1], 0) >= w[2], f"{c} waits for completion {w[2]} of {w[1]}, " \
                        f"which has completed {self.count.get(w[1], 0)} times"
                    state[c] = w
                    self.waiting[c] = (w[1], w[2])
                except StopIteration:
                    del pending[c]
                    state[c] = None
        raise AssertionError("model did not finish")


# (ring slots, Q buffers) of the kernel's instantiations: D = 128 and D = 64,
# one Q buffer on the tile path and the Gather 0 layer, two on the Scatter layer
CONFIGS = [(6, 1), (5, 2), (12, 1), (11, 2)]


@pytest.mark.parametrize("S,kqb", CONFIGS)
@pytest.mark.parametrize("seed", range(12))
def test_item_protocol_has_no_deadlock_or_parity_alias(S, kqb, seed):
    rng = random.Random(seed * 97 + S * 7 + kqb)
    rows = [rng.choice([0, 1, 1, 2, 3, 4, 7, 8]) if rng.random() < 0.85 else rng.randint(9, 40)
            for _ in range(rng.randint(1, 10))]
    Model(rows, S, kqb, rng).run()


def test_model_catches_a_short_ring():
    """The check has teeth: with a ring of 3 slots the producer's refill of
    K_j's slot no longer waits for the softmax, and some interleaving lets
    a barrier run two completions past a waiter."""
    failures = 0
    for seed in range(40):
        rng = random.Random(seed)
        rows = [rng.choice([3, 4, 7, 8, 20]) for _ in range(4)]
        try:
            Model(rows, 3, 1, rng).run()
        except AssertionError:
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("S", [6, 12])
@pytest.mark.parametrize("seed", range(12))
def test_row_protocol_with_three_gathering_warps(S, seed):
    """The single-row kernel with gathered K/V: three producer warps copy
    the tiles in turn, each waiting for its own ring slot."""
    rng = random.Random(1000 + seed * 13 + S)
    n = rng.choice([1, 2, 3, 4, 7, 16, 33, 69])
    Model([n], S, 1, rng, producers=3).run()
