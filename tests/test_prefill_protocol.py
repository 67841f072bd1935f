"""The tensor-core prefill kernels' mbarrier protocols, checked on the CPU.

Every warp role of ``gla_chunk_tc.cu`` (per-head gate) and of
``gla_chunk_tc_vec.cu`` (per-key-channel gate) is restated here as the sequence of
barrier waits and arrivals it performs per chunk (an MMA commit counts as an
arrival that happens once the MMA has run; the model lets it happen at any
later time the scheduler picks).  A randomised scheduler then advances one
role at a time, with per-role speed biases so that some roles starve while
others run ahead, and checks two properties for every chunk count and every
pattern of "wide" chunks (the explicit-decay path):

* no deadlock: every role reaches its end;
* no parity alias: an mbarrier wait names only the parity of the phase it
  wants, so a waiter must never fall two or more completed phases behind on
  the barrier it waits for (it would then wait for a phase that has already
  passed and time out).

TMA transactions and MMA commits are asynchronous: the barrier arrival lands
later, in the order the role started them.  Each role that starts them drains
them before the CTA ends, and a run may abort at any step (a bounded wait ran
out): every role then gives up at its next wait and runs only its drain; the
model checks that every role ends and that nothing is still in flight.

The model must be kept in step with the kernel: a role's steps appear in the
same order as in its source.  ``test_single_p_barrier_is_caught`` plants the
mistake of an earlier revision (one P'-ready barrier instead of one per chunk
parity) and checks that the model finds the alias it allows.
"""
import random
from collections import defaultdict

import pytest

SLOTS = 3          # gate ring depth (per-head kernel)
MASK_WARPS = 4
STATE_WARPS = 8
GATE_WARPS = 8     # per-key-channel kernel


def kernel_roles(nch, wide, single_p_barrier=False):
    """Generators of ("wait", barrier, phase) / ("arrive", barrier) /
    ("bar_sync",) steps, one per warp role of the per-head kernel (warps of a
    group are separate roles: each arrives once per barrier phase).  The MMA
    issuers: A (MMA1), B (MMA3 then MMA2), C (MMA4 into the chunk's own U)."""
    K = SLOTS
    pfull = (lambda c: ("PFull",)) if single_p_barrier else (lambda c: ("PFull", c & 1))
    pphase = (lambda c: c) if single_p_barrier else (lambda c: c >> 1)

    def producer():  # warp 0: TMA of chunks 0, 1 first; then per chunk gate sums, TMA (c >= 2)
        for c in range(min(2, nch)):
            yield ("async", ("QKFull", c & 1))  # the TMA transaction completes it
            yield ("async", ("VFull", c & 1))
        for c in range(nch):
            if c >= K:
                yield ("wait", ("GFree", c % K), c // K - 1)
            yield ("arrive", ("GReady", c % K))
            if c >= 2:
                yield ("wait", ("QKEmpty", c & 1), (c >> 1) - 1)
                yield ("async", ("QKFull", c & 1))
                yield ("wait", ("VEmpty", c & 1), (c >> 1) - 1)
                yield ("async", ("VFull", c & 1))
        yield ("drain",)  # its last copies / commits land before the CTA exits

    def issuer_a():  # warp 1: MMA1
        for c in range(nch):
            st = c & 1
            yield ("wait", ("QKFull", st), c >> 1)
            if c >= 2:
                yield ("wait", ("AFree", st), (c >> 1) - 1)
            yield ("async", ("AFull", st))
            yield ("async", ("QKEmpty", st))
        yield ("drain",)  # its last copies / commits land before the CTA exits

    def issuer_b():  # warp 2: MMA3, then MMA2
        for c in range(nch):
            st = c & 1
            yield ("wait", ("QKFull", st), c >> 1)
            yield ("wait", ("SReady",), c)
            if c >= 2:
                yield ("wait", ("OFree", st), (c >> 1) - 1)
            yield ("async", ("O3Full", st))
            yield ("async", ("SFree",))
            yield ("async", ("QKEmpty", st))
            yield ("wait", pfull(c), pphase(c))
            yield ("wait", ("VFull", st), c >> 1)
            yield ("async", ("OFull", st))
            yield ("async", ("AFree", st))
            yield ("async", ("VEmpty", st))
        yield ("drain",)  # its last copies / commits land before the CTA exits

    def issuer_c():  # warp 3: MMA4 into U of the chunk's parity
        for c in range(nch):
            st = c & 1
            yield ("wait", ("QKFull", st), c >> 1)
            yield ("wait", ("VtFull",), c)
            if c >= 2:
                yield ("wait", ("UFree", st), (c >> 1) - 1)
            yield ("async", ("UFull", st))
            yield ("async", ("VtFree",))
            yield ("async", ("QKEmpty", st))
        yield ("drain",)  # its last copies / commits land before the CTA exits

    def mask():  # warps 4..7: P' of chunk c, then the output of chunk c - 1
        for c in range(nch + 1):
            if c < nch:
                st = c & 1
                yield ("wait", ("GReady", c % K), c // K)
                yield ("wait", ("AFull", st), c >> 1)
                yield ("arrive", ("GFree", c % K))
                if wide(c):
                    yield ("wait", ("O3Full", st), c >> 1)
                yield ("arrive", pfull(c))
            if c >= 1:
                d = c - 1
                yield ("wait", ("OFull", d & 1), d >> 1)
                yield ("arrive", ("OFree", d & 1))

    def state():  # warps 8..15: split of chunk c + 1, state step c, S'_c
        for c in range(-1, nch):
            n = c + 1
            if n < nch:
                yield ("wait", ("GReady", n % K), n // K)
                yield ("wait", ("VFull", n & 1), n >> 1)
                if n >= 1:
                    yield ("wait", ("VtFree",), n - 1)
                yield ("arrive", ("VtFull",))
                yield ("arrive", ("VEmpty", n & 1))
            if c >= 0:
                yield ("wait", ("UFull", c & 1), c >> 1)
                yield ("arrive", ("UFree", c & 1))
            if n < nch:
                if c >= 0:
                    yield ("wait", ("SFree",), c)
                yield ("arrive", ("SReady",))
            if c >= 0:
                yield ("arrive", ("GFree", c % K))

    roles = {"producer": producer(), "issuer_a": issuer_a(), "issuer_b": issuer_b(),
             "issuer_c": issuer_c()}
    for w in range(MASK_WARPS):
        roles[f"mask{w}"] = mask()
    for w in range(STATE_WARPS):
        roles[f"state{w}"] = state()
    return roles


def arrival_counts():
    """Arrivals per phase of the per-head kernel's barriers (default 1)."""
    n = {("QKEmpty", 0): 3, ("QKEmpty", 1): 3, ("PFull",): MASK_WARPS, ("PFull", 0): MASK_WARPS,
         ("PFull", 1): MASK_WARPS, ("OFree", 0): MASK_WARPS, ("OFree", 1): MASK_WARPS,
         ("VEmpty", 0): 1 + STATE_WARPS, ("VEmpty", 1): 1 + STATE_WARPS,
         ("UFree", 0): STATE_WARPS, ("UFree", 1): STATE_WARPS, ("VtFull",): STATE_WARPS,
         ("SReady",): STATE_WARPS}
    for i in range(SLOTS):
        n[("GFree", i)] = MASK_WARPS + STATE_WARPS
    return n


def vector_kernel_roles(nch, wide, tokens_in_wide_chunk=2, mix=False):
    """The per-key-channel kernel.  Chunks the gate group finds "wide" are
    processed by it token by token (one group barrier per token) and skip the
    MMAs; the others run the tensor-core path.  The gate group's barrier is an
    mbarrier whose phases the warps count themselves.  With ``mix`` (the
    mixer's steps inside the kernel) the mask warps read each chunk's Q' and
    Kt rows and release the Q/K buffer too."""
    def producer():  # warp 0, lane 0
        for c in range(nch):
            if c >= 1:
                yield ("wait", ("GEmpty",), c - 1)
            yield ("async", ("GFull",))
            if c >= 1:
                yield ("wait", ("QKEmpty",), c - 1)
            yield ("async", ("QKFull",))
            if c >= 1:
                yield ("wait", ("VEmpty",), c - 1)
            yield ("async", ("VFull",))
        yield ("drain",)  # its last copies / commits land before the CTA exits

    def issuer():  # warp 1, lane 0: MMA1, MMA3, MMA4, MMA2 per tensor-core chunk
        n = 0
        for c in range(nch):
            yield ("wait", ("Scaled", c & 1), c >> 1)
            yield ("arrive", ("Ack", c & 1))
            if wide(c):
                continue
            yield ("async", ("AFull",))
            yield ("wait", ("SbReady",), n)
            if n >= 2:
                yield ("wait", ("OFree", n & 1), (n >> 1) - 1)
            yield ("wait", ("VFull",), c)
            yield ("async", ("SFull",))
            yield ("async", ("QKEmpty",))
            yield ("wait", ("PFull", n & 1), n >> 1)
            yield ("async", ("OFull", n & 1))
            yield ("async", ("VEmpty",))
            n += 1
        yield ("drain",)  # its last copies / commits land before the CTA exits

    def mask():  # warps 4..7
        n, pending = 0, False
        for c in range(nch + 1):
            tc = False
            if c < nch:
                yield ("wait", ("Scaled", c & 1), c >> 1)
                yield ("arrive", ("Ack", c & 1))
                tc = not wide(c)
                if mix:
                    yield ("arrive", ("QKEmpty",))
                if tc:
                    yield ("wait", ("AFull",), n)
                    yield ("arrive", ("PFull", n & 1))
            if pending:
                m = n - 1
                yield ("wait", ("OFull", m & 1), m >> 1)
                yield ("arrive", ("OFree", m & 1))
            pending = tc
            if tc:
                n += 1

    def gate(first):  # warps 8..15
        k = 0  # group barrier phases

        def group_sync():
            nonlocal k
            yield ("arrive", ("GateSync",))
            yield ("wait", ("GateSync",), k)
            k += 1

        n, last_tc = 0, False
        for c in range(nch):
            yield ("wait", ("GFull",), c)
            yield from group_sync()          # partial sums written
            yield from group_sync()          # wide vote
            if c >= 2:
                yield ("wait", ("Ack", c & 1), (c - 2) >> 1)
            if not wide(c):
                if last_tc:                  # the state pass first
                    yield ("wait", ("SFull",), n - 1)
                yield ("arrive", ("SbReady",))
                yield ("wait", ("QKFull",), c)
                yield from group_sync()      # done with g
                if first:
                    yield ("arrive", ("GEmpty",))
                yield ("arrive", ("Scaled", c & 1))
                last_tc = True
                n += 1
            else:
                yield ("wait", ("QKFull",), c)
                yield ("arrive", ("Scaled", c & 1))
                if last_tc:
                    yield ("wait", ("SFull",), n - 1)
                yield ("wait", ("VFull",), c)
                for _ in range(tokens_in_wide_chunk):
                    yield from group_sync()
                yield from group_sync()      # done with g, Q, K, V
                if first:
                    yield ("arrive", ("GEmpty",))
                    yield ("arrive", ("QKEmpty",))
                    yield ("arrive", ("VEmpty",))
                last_tc = False
        if last_tc:
            yield ("wait", ("SFull",), n - 1)

    roles = {"producer": producer(), "issuer": issuer()}
    for w in range(MASK_WARPS):
        roles[f"mask{w}"] = mask()
    for w in range(GATE_WARPS):
        roles[f"gate{w}"] = gate(w == 0)
    return roles


def vector_arrival_counts(mix=False):
    n = {("QKEmpty",): 1 + MASK_WARPS if mix else 1,
         ("Scaled", 0): GATE_WARPS, ("Scaled", 1): GATE_WARPS, ("SbReady",): GATE_WARPS,
         ("GateSync",): GATE_WARPS, ("PFull", 0): MASK_WARPS, ("PFull", 1): MASK_WARPS,
         ("OFree", 0): MASK_WARPS, ("OFree", 1): MASK_WARPS,
         ("Ack", 0): 1 + MASK_WARPS, ("Ack", 1): 1 + MASK_WARPS}
    return n


def run_schedule(nch, wide, seed, vector=False, roles=None, need=None, abort_at=None,
                 drain_on_abort=True, **kw):
    """Returns None when every role finishes, else a description of the fault.

    ("async", bar) steps are the TMA transactions and MMA commits a role starts:
    the barrier arrival happens later, at a time the scheduler picks, in the
    order the role started them (one thread's commits complete in order).
    ("drain",) waits until the role's own started operations have all landed.
    With ``abort_at``, a bounded wait runs out after that many scheduler steps:
    from then on every role gives up at its next wait (as the kernels' waits do
    once the abort flag is set) and runs only its teardown, a drain for the
    roles that start asynchronous operations.  Every role must reach the end
    with no operation of its own still in flight."""
    rnd = random.Random(seed)
    if roles is None:
        roles = (vector_kernel_roles if vector else kernel_roles)(nch, wide, **kw)
        need = vector_arrival_counts(kw.get("mix", False)) if vector else arrival_counts()
    pending, done = defaultdict(int), defaultdict(int)
    inflight = defaultdict(list)  # role -> barriers of its started operations, oldest first
    step = {n: next(g, None) for n, g in roles.items()}
    speed = {n: rnd.choice([0.02, 1.0, 1.0, 8.0]) for n in roles}
    in_bar_sync = set()
    aborted, nsteps = False, 0

    def arrive(bar):
        pending[bar] += 1
        if pending[bar] == need.get(bar, 1):
            pending[bar] = 0
            done[bar] += 1

    def teardown(n):
        if drain_on_abort:
            yield ("drain",)

    while True:
        if abort_at is not None and not aborted and nsteps >= abort_at:
            aborted = True
        if aborted:
            for n in list(step):
                s = step[n]
                if s is not None and s[0] in ("wait", "bar_sync"):
                    roles[n] = teardown(n)
                    step[n] = next(roles[n], None)
                    in_bar_sync.discard(n)
        live = [n for n in step if step[n] is not None]
        landing = [n for n in inflight if inflight[n]]
        if not live:
            if landing:
                return "end with operations in flight: " + ", ".join(landing)
            return None
        if len(in_bar_sync) == STATE_WARPS:
            for n in in_bar_sync:
                step[n] = next(roles[n], None)
            in_bar_sync.clear()
            continue
        ready = []
        for n in live:
            s = step[n]
            if s[0] == "wait":
                if done[s[1]] > s[2] + 1:
                    return f"alias: {n} waits for phase {s[2]} of {s[1]}, {done[s[1]]} completed"
                if done[s[1]] > s[2]:
                    ready.append(n)
            elif s[0] == "drain":
                if not inflight[n]:
                    ready.append(n)
            elif s[0] in ("arrive", "async") or n not in in_bar_sync:
                ready.append(n)
        if not ready and not landing:
            return "deadlock: " + ", ".join(f"{n} at {step[n]}" for n in live)
        nsteps += 1
        choices = ready + [("land", m) for m in landing]
        weights = [speed[m] for m in ready] + [1.0] * len(landing)
        pick = rnd.choices(choices, weights=weights)[0]
        if isinstance(pick, tuple):
            arrive(inflight[pick[1]].pop(0))
            continue
        n = pick
        s = step[n]
        if s[0] == "bar_sync":
            in_bar_sync.add(n)
            continue
        if s[0] == "arrive":
            arrive(s[1])
        elif s[0] == "async":
            inflight[n].append(s[1])
        step[n] = next(roles[n], None)


WIDE_PATTERNS = {
    "none": lambda c: False,
    "all": lambda c: True,
    "odd": lambda c: c % 2 == 1,
    "every_third": lambda c: c % 3 == 0,
}


@pytest.mark.parametrize("pattern", sorted(WIDE_PATTERNS))
def test_protocol_has_no_deadlock_or_alias(pattern):
    wide = WIDE_PATTERNS[pattern]
    for nch in range(0, 9):
        for seed in range(150):
            fault = run_schedule(nch, wide, seed)
            assert fault is None, f"{nch} chunks, seed {seed}: {fault}"


@pytest.mark.parametrize("mix", [False, True], ids=["plain", "mixer"])
@pytest.mark.parametrize("pattern", sorted(WIDE_PATTERNS) + ["first_two", "runs"])
def test_vector_protocol_has_no_deadlock_or_alias(pattern, mix):
    extra = {"first_two": lambda c: c < 2, "runs": lambda c: (c // 3) % 2 == 1}
    wide = WIDE_PATTERNS.get(pattern) or extra[pattern]
    for nch in range(0, 9):
        for seed in range(120):
            fault = run_schedule(nch, wide, seed, vector=True, mix=mix)
            assert fault is None, f"{nch} chunks, seed {seed}: {fault}"


def test_single_p_barrier_is_caught():
    faults = [run_schedule(nch, WIDE_PATTERNS["none"], seed, single_p_barrier=True)
              for nch in range(2, 6) for seed in range(200)]
    assert any(f is not None and f.startswith("alias") and "PFull" in f for f in faults)


@pytest.mark.parametrize("vector", [False, True], ids=["per_head", "per_key_channel"])
def test_abort_drains_and_ends(vector):
    """A wait that runs out at any point: every role ends, each with its own
    copies and MMA commits landed (the drain), and none waits on another."""
    for pattern in ("none", "odd"):
        wide = WIDE_PATTERNS[pattern]
        for nch in range(1, 7):
            for seed in range(60):
                abort_at = random.Random(1000 + seed).randrange(0, 40 * nch + 20)
                fault = run_schedule(nch, wide, seed, vector=vector, abort_at=abort_at)
                assert fault is None, f"{pattern}, {nch} chunks, seed {seed}, abort at {abort_at}: {fault}"


def test_abort_without_drain_is_caught():
    """The planted mistake: a teardown that only waits out a fixed time (no
    drain) lets a CTA end with a copy or a commit still in flight."""
    faults = [run_schedule(nch, WIDE_PATTERNS["none"], seed, abort_at=ab, drain_on_abort=False)
              for nch in range(2, 5) for seed in range(40) for ab in (5, 15, 30)]
    assert any(f is not None and f.startswith("end with operations in flight") for f in faults)
