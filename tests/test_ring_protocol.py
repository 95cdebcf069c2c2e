"""Model check of the fused kernel's ring-release protocols (host logic, no
GPU).

The producer, the UMMA issuer, the tensor pipe (which completes commits in
issue order, at any later time) and the promotion epilogue are simulated as
agents over mbarriers with the hardware's parity semantics: a barrier counts
completed phases, and a wait for parity P succeeds once the phase with that
parity has completed, i.e. while (completed phases & 1) != P.  Random
interleavings must never deadlock, never let the producer overwrite a stage
whose UMMAs are still pending, and never let the UMMAs read a stage before
the producer filled it for that iteration.

Modelled: stages released per commit in groups of CG (one commit on the
group's barrier after the group's last stage), and, for promotion kernels,
stages freed by the per-K-block accumulator commit that the epilogue also
waits on (safe while the ring depth S is at most the number of accumulator
buffers NB).  The ring position is kept with counters, as the kernel does.
"""
import random

import pytest


class Ring:
    """Stage, its use parity, index in group, group slot, its use parity."""

    def __init__(self):
        self.s = self.ph = self.gi = self.gs = self.gph = 0

    def next(self, S, CG, NG):
        self.s += 1
        if self.s == S:
            self.s, self.ph = 0, self.ph ^ 1
        self.gi += 1
        if self.gi == CG:
            self.gi = 0
            self.gs += 1
            if self.gs == NG:
                self.gs, self.gph = 0, self.gph ^ 1


def passes(count, parity):
    return (count & 1) != parity


def simulate(S, CG, T, acc_release=False, NB=4, seed=0, promote=None, early_commit=False):
    """Run T ring iterations; return None, or a string naming the violation.
    early_commit plants a bug: the group's commit after its first stage."""
    promote = acc_release if promote is None else promote
    rng = random.Random(seed)
    NG = S // CG
    full = [0] * S            # completed phases
    empty = [0] * NG
    tfull = [0] * NB
    tempty = [0] * NB
    content = [None] * S      # iteration whose data the stage holds
    pending = {}              # stage -> iteration whose UMMAs have not completed
    pipe = []                 # issued, not completed: ("umma", s, g) / ("commit", kind, idx)
    prod, mma, epi = Ring(), Ring(), 0
    gp = gm = 0

    def prod_step():
        nonlocal gp
        if gp >= T:
            return False
        if acc_release:
            if gp >= S:
                j = gp - S
                if not passes(tfull[j % NB], (j // NB) & 1):
                    return False
        elif not passes(empty[prod.gs], prod.gph ^ 1):
            return False
        s = prod.s
        if s in pending:
            raise AssertionError(f"stage {s} overwritten for iteration {gp} while the UMMAs "
                                 f"of iteration {pending[s]} are pending")
        content[s] = gp
        full[s] += 1
        prod.next(S, CG, NG)
        gp += 1
        return True

    def mma_step():
        nonlocal gm
        if gm >= T:
            return False
        b = gm % NB
        if promote and not passes(tempty[b], ((gm // NB) & 1) ^ 1):
            return False
        s = mma.s
        if not passes(full[s], mma.ph):
            return False
        if content[s] != gm:
            raise AssertionError(f"iteration {gm} read stage {s} holding iteration {content[s]}")
        pending[s] = gm
        pipe.append(("umma", s, gm))
        if not acc_release and mma.gi == (0 if early_commit else CG - 1):
            pipe.append(("commit", "empty", mma.gs))
        if promote:
            pipe.append(("commit", "tfull", b))
        mma.next(S, CG, NG)
        gm += 1
        return True

    def pipe_step():
        if not pipe:
            return False
        kind, a, c = pipe.pop(0)
        if kind == "umma":
            if pending.get(a) == c:
                del pending[a]
        elif a == "empty":
            empty[c] += 1
        else:
            tfull[c] += 1
        return True

    def epi_step():
        nonlocal epi
        if not promote or epi >= T:
            return False
        b = epi % NB
        if not passes(tfull[b], (epi // NB) & 1):
            return False
        tempty[b] += 1
        epi += 1
        return True

    agents = [prod_step, mma_step, pipe_step, epi_step]
    while gp < T or gm < T or pipe or (promote and epi < T):
        order = agents[:]
        rng.shuffle(order)
        # bias towards slow completion sometimes, so the issuer runs ahead
        if rng.random() < 0.5:
            order.sort(key=lambda f: f is pipe_step)
        if not any(f() for f in order[:1]) and not any(f() for f in order):
            return f"deadlock at producer {gp}, issuer {gm}, epilogue {epi}"
    return None


@pytest.mark.parametrize("S,CG", [(2, 1), (3, 1), (4, 1), (4, 2), (5, 1), (6, 2), (6, 3),
                                  (8, 2), (8, 4)])
def test_grouped_stage_release(S, CG):
    for seed in range(40):
        assert simulate(S, CG, T=61, seed=seed) is None


@pytest.mark.parametrize("S,NB", [(2, 4), (3, 4), (4, 4), (2, 2)])
def test_release_by_accumulator_commit(S, NB):
    """Promotion kernels: the stage (or INT8 operand slot, three of them) of
    K block g is freed by block g's accumulator commit (four buffers, or two
    for 256-wide tiles, the epilogue draining them in order)."""
    for seed in range(40):
        assert simulate(S, 1, T=53, acc_release=True, NB=NB, seed=seed) is None


def test_release_by_accumulator_commit_needs_enough_buffers():
    """A ring deeper than the accumulator buffers breaks the release by the
    accumulator commit (the host allows it only up to the buffer count)."""
    bad = 0
    for seed in range(200):
        try:
            if simulate(4, 1, T=53, acc_release=True, NB=2, seed=seed) is not None:
                bad += 1
        except AssertionError:
            bad += 1
    assert bad > 0


def test_per_stage_release_with_promotion():
    """The same epilogue handshake with per-stage commits (deeper rings)."""
    for seed in range(40):
        assert simulate(6, 1, T=47, acc_release=False, promote=True, seed=seed) is None


def test_model_catches_a_broken_release():
    """The check has teeth: committing a group after its first stage instead
    of its last frees stages whose UMMAs are still pending; some interleaving
    overwrites one (or the producer and issuer deadlock)."""
    bad = 0
    for seed in range(200):
        try:
            if simulate(4, 2, T=53, seed=seed, early_commit=True) is not None:
                bad += 1
        except AssertionError:
            bad += 1
    assert bad > 0
