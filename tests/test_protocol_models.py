"""CPU models of two synchronisation protocols in the int8-operand kernels
(gemm_s8.cu), restated from the kernels' rules.  They test the protocols'
logic, not the kernels.

1. The few-token kernel's ring.  A producer fills S slots in order.  Two
   converter warpgroups take alternate stages, and one MMA thread consumes
   stages in order.  Copies complete out of order.  mbarrier parity waits
   return as soon as the barrier's completed-phase count has the other
   parity.  With one full barrier per slot and an odd S, a group can pass
   its wait before its own copy landed: it was waiting on every other phase
   only.  With one full barrier per slot and converter group, as the kernel
   has, it cannot.

2. The wide-token kernel's rotating accumulator regions.  P token parts
   share P + 1 regions, and each part moves into the free region at the
   end of its chunk.  The MMA thread's commits and the epilogue's replayed
   folds must visit the same regions in the same order.  No two parts may
   hold one region, and every chunk must stay within 1024 K.
"""
import random

import pytest

CHUNK_STAGES = 16  # 64-K stages per 1024-K chunk in the wide kernel


class Barrier:
    """An mbarrier: an arrival count and a transaction count per phase."""

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.completed = 0

    def try_wait(self, parity):
        return (self.completed & 1) != parity

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        self._check()

    def complete_tx(self, n):
        self.tx -= n
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count


def run_ring(S, n, groups, per_group, seed):
    """One CTA's stages through the ring; returns 'ok' or what went wrong."""
    rnd = random.Random(seed)
    full8 = [Barrier(1) for _ in range(groups * S if per_group else S)]
    full16 = [Barrier(4) for _ in range(S)]
    empty = [Barrier(1) for _ in range(S)]
    landed = [None] * S      # the stage whose bytes the slot holds
    tmem = [None] * S        # the stage widened into the tensor-memory stage
    inflight = []
    produced, consumed = 0, 0
    conv = [{"ks": g, "uses": 0} for g in range(groups)]
    for _ in range(100000):
        if consumed == n:
            return "ok"
        rnd.shuffle(inflight)  # copies land in any order
        keep = []
        for due, s, ks, bar in inflight:
            if due <= 0:
                landed[s] = ks
                bar.complete_tx(1)
            else:
                keep.append((due - 1, s, ks, bar))
        inflight = keep
        if produced < n:
            s = produced % S
            if produced < S or empty[s].try_wait(((produced // S) & 1) ^ 1):
                bar = full8[(produced % groups) * S + s] if per_group else full8[s]
                bar.arrive(tx=1)
                inflight.append((rnd.choice([0, 1, 2, 4, 20, 60]), s, produced, bar))
                produced += 1
        for g, c in enumerate(conv):
            ks = c["ks"]
            if ks >= n:
                continue
            s = ks % S
            if per_group:
                bar, parity = full8[g * S + s], (c["uses"] >> s) & 1
            else:
                bar, parity = full8[s], (ks // S) & 1
            if bar.try_wait(parity):
                if landed[s] != ks:
                    return "early pass"
                if per_group:
                    c["uses"] ^= 1 << s
                tmem[s] = ks
                for _ in range(4):
                    full16[s].arrive()
                c["ks"] += groups
        s = consumed % S
        if full16[s].try_wait((consumed // S) & 1):
            if tmem[s] != consumed:
                return "wrong stage"
            empty[s].arrive()
            consumed += 1
    return "stall"


@pytest.mark.parametrize("S", [5, 7])
def test_one_full_barrier_per_slot_passes_early_with_an_odd_ring(S):
    results = {run_ring(S, 60, 2, False, seed) for seed in range(200)}
    assert "early pass" in results


@pytest.mark.parametrize("S,groups", [(4, 2), (5, 2), (6, 2), (7, 2), (5, 3)])
def test_a_full_barrier_per_slot_and_group_never_passes_early(S, groups):
    for seed in range(200):
        assert run_ring(S, 60, groups, True, seed) == "ok"


def chunk_start(P, q, j):
    return j == 0 or (j + q * (CHUNK_STAGES // P)) % CHUNK_STAGES == 0


def part_starting(P, j):
    for q in range(P):
        if (j + q * (CHUNK_STAGES // P)) % CHUNK_STAGES == 0:
            return q
    return -1


def chunks(P, q, n):
    return sum(1 for j in range(n) if chunk_start(P, q, j))


@pytest.mark.parametrize("P", [2, 3, 4])
@pytest.mark.parametrize("units", [[1], [5], [8], [17], [80, 80], [2, 300, 3], [1024]])
def test_rotating_regions_commit_and_fold_in_the_same_order(P, units):
    # the MMA thread: commits at chunk ends, moves the part into the free region
    table, free = list(range(P)), P
    commits = []
    for n in units:
        start = [0] * P
        for j in range(1, n):
            q = part_starting(P, j)
            if q < 0:
                continue
            assert j - start[q] <= CHUNK_STAGES
            commits.append((table[q], q))
            table[q], free = free, table[q]
            start[q] = j
            assert len(set(table)) == P and free not in table
        for q in range(P):
            assert n - start[q] <= CHUNK_STAGES
            commits.append((table[q], q))
    # the epilogue: replays the same table and folds in the same order
    table, free = list(range(P)), P
    folds = []
    for n in units:
        for j in range(1, n):
            q = part_starting(P, j)
            if q >= 0:
                folds.append((table[q], q))
                table[q], free = free, table[q]
        for q in range(P):
            folds.append((table[q], q))
    assert folds == commits
    assert len(folds) == sum(chunks(P, q, n) for n in units for q in range(P))
    # after stage 0 no two parts end a chunk at the same stage
    for j in range(1, 64):
        assert sum(1 for q in range(P) if chunk_start(P, q, j)) <= 1
