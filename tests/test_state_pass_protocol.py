"""Model check of the synchronisation protocol of the tensor-core state pass (CPU only).

chunk_state_tc_kernel (kda_gated_delta_gb300/csrc/kda_prefill.cu) runs its chunk loop as separate
warp roles that hand work to each other through mbarriers: the Delta pass, the S update, the Z /
W' / output warps, two MMA issuers and a copy warp.  A mistake in that protocol shows up on the
GPU only as a bounded wait that gives up (device error 3) or as silently wrong operands.  This
test replays the protocol, role by role and wait by wait as the kernel orders them, under many
random interleavings:

  * a parity wait (mbarrier.try_wait.parity) completes when the phase it names has completed and
    no later phase has; a waiter that could see the barrier two phases ahead is an error;
  * each issuer's MMAs execute in issue order, the two issuers' MMAs interleave freely, and a
    commit arrives once all of its issuer's earlier MMAs have executed; copies land in any order;
  * every operand an MMA or a warp reads must hold the chunk's version the algorithm needs when it
    is read (no buffer reused too early);
  * the run must finish (no deadlock), and the copy warp's closing drain must leave no copy in
    flight when that warp exits.

The model has to be kept in step with the kernel by hand: it mirrors the kernel's wait lists,
buffer indices and arrival counts, not its arithmetic.
"""
import random

import pytest


class Bar:
    def __init__(self, name, count=1):
        self.name, self.count, self.pend, self.phase = name, count, 0, 0

    def arrive(self, n=1):
        for _ in range(n):
            self.pend += 1
            if self.pend == self.count:
                self.pend = 0
                self.phase += 1


def last_phase(n, s, depth):
    """Phase of ring slot s after n copies: it last received chunk s + depth ((n - 1 - s) // depth)."""
    return (n - 1 - s) // depth


class Model:
    def __init__(self, n, seed, single_delta_barrier=False, drain_phase=last_phase):
        self.n, self.rng = n, random.Random(seed)
        self.drain_phase = drain_phase
        self.w = [Bar(f"w{i}") for i in range(4)]
        self.kt = [Bar(f"kt{i}") for i in range(3)]
        self.u = [Bar(f"u{i}") for i in range(2)]
        self.qp = [Bar("qp0"), Bar("qp1")]
        self.chain, self.c, self.z = Bar("chain"), Bar("c"), Bar("z")
        self.o = [Bar("o0"), Bar("o1")]
        if single_delta_barrier:        # the variant with one Delta-ready barrier: must be caught
            d = Bar("delta", 128)
            self.delta = [d, d]
        else:
            self.delta = [Bar("delta0", 128), Bar("delta1", 128)]
        self.single = single_delta_barrier
        self.sh = [Bar(f"sh{i}", 256) for i in range(4)]
        self.zw = [Bar(f"zw{i}", 128) for i in range(4)]
        self.dz_free, self.do_free = Bar("dz_free", 128), Bar("do_free", 128)
        self.mem = {}
        self.pipe = {0: [], 1: []}
        self.issued = {0: 0, 1: 0}
        self.executed = {0: 0, 1: 0}
        self.commits = []
        self.copies = []

    # ---- effects
    def read(self, res, tag, who):
        got = self.mem.get(res)
        assert got == tag, f"{who} read {res}: expected {tag}, found {got}"

    def write(self, res, tag):
        self.mem[res] = tag

    def mma(self, issuer, reads, writes):
        self.pipe[issuer].append((reads, writes))
        self.issued[issuer] += 1

    def commit(self, issuer, bar):
        self.commits.append((issuer, self.issued[issuer], bar))

    def copy(self, dst, bar):
        self.copies.append((dst, bar))

    # ---- waits: (barrier, parity, phase the waiter means)
    def delta_wait(self, i):
        if self.single:
            return (self.delta[0], i & 1, i)
        return (self.delta[i & 1], (i >> 1) & 1, i >> 1)


def ring(bars, j, depth):
    return (bars[j % depth], (j // depth) & 1, j // depth)


def single(bar, k):
    return (bar, k & 1, k)


# ---- the roles, in the kernel's order of waits
def chain_and_c_issuer(M):            # warp 16
    n = M.n
    yield ring(M.sh, 0, 4)
    yield ring(M.w, 0, 4)
    M.mma(0, [("SH0", "S0"), ("W0", "W0")], [("DA", "A0")])
    M.commit(0, M.chain)
    for i in range(n):
        yield M.delta_wait(i)
        yield ring(M.sh, i, 4)
        if i + 1 < n:
            yield ring(M.zw, i, 4)                   # Z_{i+1} and W'_{i+1}
            M.mma(0, [(f"SH{i & 1}", f"S{i}"), (f"W{(i + 1) & 3}", f"W'{i + 1}"), (f"DH{i & 1}", f"D{i}"),
                      (f"Z{(i + 1) & 1}", f"Z{i + 1}")], [("DA", f"A{i + 1}")])
            M.commit(0, M.chain)
        yield ring(M.kt, i, 3)
        M.mma(0, [(f"DH{i & 1}", f"D{i}"), (f"KT{i % 3}", f"K{i}")], [("DC", f"C{i}")])
        M.commit(0, M.c)


def z_and_output_issuer(M):           # warp 17
    n = M.n

    def issue_z(m):
        yield ring(M.w, m, 4)
        yield ring(M.kt, m - 1, 3)
        if m >= 2:
            yield single(M.dz_free, m - 2)
        M.mma(1, [(f"W{m & 3}", f"W{m}"), (f"KT{(m - 1) % 3}", f"K{m - 1}")], [("DZ", f"Z{m}")])
        M.commit(1, M.z)

    if n >= 2:
        yield from issue_z(1)
    for i in range(n):
        if i + 2 < n:
            yield from issue_z(i + 2)
        yield M.delta_wait(i)
        yield ring(M.sh, i, 4)
        yield ring(M.qp, i, 2)
        if i >= 1:
            yield single(M.do_free, i - 1)
        M.mma(1, [(f"DH{i & 1}", f"D{i}"), (f"SH{i & 1}", f"S{i}"), (f"QP{i & 1}", f"QP{i}")], [("DO", f"O{i}")])
        M.commit(1, M.o[i & 1])


def copy_warp(M):                     # warp 18
    n = M.n

    def w(j): M.copy({f"W{j & 3}": f"W{j}"}, M.w[j & 3])
    def kt(j): M.copy({f"KT{j % 3}": f"K{j}", f"G{j % 3}": f"G{j}"}, M.kt[j % 3])
    def u(j): M.copy({f"U{j & 1}": f"U{j}"}, M.u[j & 1])
    def qp(j): M.copy({f"QP{j & 1}": f"QP{j}"}, M.qp[j & 1])

    for j in range(min(4, n)):
        w(j)
    for j in range(min(2, n)):
        kt(j)
        u(j)
        qp(j)
    for i in range(n):
        yield M.delta_wait(i)
        if i + 2 < n:
            u(i + 2)
        if i + 4 < n:
            w(i + 4)
        if i + 2 < n:
            if i >= 1:
                yield ring(M.sh, i, 4)
                yield ring(M.zw, i - 1, 4)
            kt(i + 2)
        if i + 2 < n:
            yield ring(M.o, i, 2)
            qp(i + 2)
    # drain: the copies still in flight land before the CTA exits
    for bars, depth in ((M.w, 4), (M.kt, 3), (M.u, 2), (M.qp, 2)):
        for s in range(min(depth, n)):
            ph = M.drain_phase(n, s, depth)
            yield (bars[s], ph & 1, ph)


def delta_pass(M):                    # warps 0..3
    for j in range(M.n):
        yield single(M.chain, j)
        if j >= 2:
            yield ring(M.o, j - 2, 2)
        yield ring(M.u, j, 2)
        M.read("DA", f"A{j}", "Delta pass")
        M.read(f"U{j & 1}", f"U{j}", "Delta pass")
        M.write(f"DH{j & 1}", f"D{j}")
        M.delta[j & 1].arrive(128)


def state_update(M):                  # warps 4..11
    M.write("SH0", "S0")
    M.sh[0].arrive(256)
    for j in range(M.n):
        yield single(M.c, j)
        yield ring(M.kt, j, 3)
        if j >= 1:
            yield ring(M.o, j - 1, 2)
        M.read("DC", f"C{j}", "S update")
        M.read(f"G{j % 3}", f"G{j}", "S update")
        if j + 1 < M.n:
            M.write(f"SH{(j + 1) & 1}", f"S{j + 1}")
        M.sh[(j + 1) & 3].arrive(256)


def z_w_output_warps(M):              # warps 12..15
    n = M.n

    def z_epilogue(m):
        yield single(M.z, m - 1)
        if m >= 2:
            yield M.delta_wait(m - 2)            # the Z slot's previous reader, chain MMA m - 2, is done
        yield ring(M.w, m, 4)
        yield ring(M.kt, m - 1, 3)
        M.read("DZ", f"Z{m}", "Z epilogue")
        M.write(f"Z{m & 1}", f"Z{m}")
        M.dz_free.arrive(128)
        M.read(f"W{m & 3}", f"W{m}", "W' scaling")
        M.read(f"G{(m - 1) % 3}", f"G{m - 1}", "W' scaling")
        M.write(f"W{m & 3}", f"W'{m}")
        M.zw[(m - 1) & 3].arrive(128)

    if n >= 2:
        yield from z_epilogue(1)
    for i in range(n):
        if i + 2 < n:
            yield from z_epilogue(i + 2)
        yield ring(M.o, i, 2)
        M.read("DO", f"O{i}", "output copy")
        M.do_free.arrive(128)


def run(n, seed, single_delta_barrier=False, drain_phase=last_phase):
    M = Model(n, seed, single_delta_barrier, drain_phase)
    roles = {"chain+(c)": chain_and_c_issuer(M), "Z+out": z_and_output_issuer(M), "copies": copy_warp(M),
             "Delta": delta_pass(M), "S": state_update(M), "Z/W'/out warps": z_w_output_warps(M)}
    waiting, done = {}, set()

    def step(k):
        try:
            waiting[k] = next(roles[k])
        except StopIteration:
            done.add(k)
            if k == "copies":
                assert not M.copies, f"the copy warp exits with {len(M.copies)} copies in flight"

    for k in roles:
        step(k)
    for _ in range(400000):
        if len(done) == len(roles) and not any(M.pipe.values()) and not M.copies and not M.commits:
            return
        moves = []
        for k in roles:
            if k in done:
                continue
            bar, parity, phase = waiting[k]
            assert bar.phase <= phase + 1, f"{k} waits for phase {phase} of {bar.name}, which is at {bar.phase}"
            if (bar.phase & 1) != parity:
                moves.append(("role", k))
        moves += [("mma", q) for q in M.pipe if M.pipe[q]]
        moves += [("copy", i) for i in range(len(M.copies))]
        moves += [("commit", i) for i, (q, cnt, _) in enumerate(M.commits) if M.executed[q] >= cnt]
        assert moves, "deadlock: " + ", ".join(
            f"{k} on {waiting[k][0].name} phase {waiting[k][2]}" for k in roles if k not in done)
        kind, x = M.rng.choice(moves)
        if kind == "role":
            step(x)
        elif kind == "mma":
            reads, writes = M.pipe[x].pop(0)
            for r, t in reads:
                M.read(r, t, f"MMA of issuer {x}")
            for r, t in writes:
                M.write(r, t)
            M.executed[x] += 1
        elif kind == "copy":
            dst, bar = M.copies.pop(x)
            for r, t in dst.items():
                M.write(r, t)
            bar.arrive()
        else:
            _, _, bar = M.commits.pop(x)
            bar.arrive()
    raise AssertionError("no progress")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 9, 17, 40])
def test_protocol_random_schedules(n):
    for seed in range(60):
        run(n, seed)


def test_single_delta_barrier_is_caught():
    """One Delta-ready barrier instead of two: its late consumers could see it two phases ahead."""
    failures = 0
    for seed in range(60):
        try:
            run(5, seed, single_delta_barrier=True)
        except AssertionError:
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("wrong", [lambda n, s, d: (n - s) // d, lambda n, s, d: (n - 1 - s) // d - 1])
def test_wrong_drain_phase_is_caught(wrong):
    """A drain that waits one phase too far never ends; one that waits one phase too early lets
    the copy warp exit with its last copies in flight."""
    failures = 0
    for n in (1, 3, 5, 8):
        for seed in range(10):
            try:
                run(n, seed, drain_phase=wrong)
            except AssertionError:
                failures += 1
    assert failures > 0


def _kernel_barriers():
    """Barrier name -> arrival count per slot, read from chunk_state_tc_kernel's initialisation."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "kda_gated_delta_gb300", "csrc", "kda_prefill.cu")).read()
    body = src[src.index("chunk_state_tc_kernel(const StateArgs a)"):]
    block = body[:body.index("tc::fence_mbar_init();")]
    block = block[block.rindex("if (tid == 0) {"):]
    bars = {}
    # statements, with "for (int i = 0; i < N; ++i) { ... }" or a single statement after it expanded
    for m in re.finditer(r"for \(int i = 0; i < (\d+); \+\+i\) (\{[^}]*\}|[^;]*;)", block):
        n = int(m.group(1))
        for name, count in re.findall(r"mbar_init\(&bars->(\w+)\[i\], (\d+)\)", m.group(2)):
            bars[name] = [int(count)] * n
    rest = re.sub(r"for \(int i = 0; i < \d+; \+\+i\) (\{[^}]*\}|[^;]*;)", "", block)
    for name, idx, count in re.findall(r"mbar_init\(&bars->(\w+)(?:\[(\d+)\])?, (\d+)\)", rest):
        if idx:
            slots = bars.setdefault(name, [])
            assert int(idx) == len(slots), (name, idx)
            slots.append(int(count))
        else:
            bars[name] = int(count)
    return bars


def test_model_mirrors_the_kernel_barriers():
    """The model's barriers have the kernel's ring depths and arrival counts (the issuers' drain
    barriers, used once after the loop, are not part of the chunk protocol)."""
    k = _kernel_barriers()
    M = Model(1, 0)
    names = {"w": "w", "kt": "kt", "u": "u", "qp": "qp", "o": "o", "delta_ready": "delta", "sh_ready": "sh",
             "zw_ready": "zw", "chain": "chain", "c": "c", "z": "z", "dz_free": "dz_free", "do_free": "do_free"}
    assert set(k) - {"drain"} == set(names), sorted(k)
    for kname, mname in names.items():
        mb = getattr(M, mname)
        got = [b.count for b in mb] if isinstance(mb, list) else mb.count
        assert got == k[kname], (kname, got, k[kname])
