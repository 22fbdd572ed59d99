"""Model check of the tensor-core contraction kernel's mbarrier protocol
(bit_expert_matvec_moe_b300/csrc/moe_tc.cu, tc_contract_kernel): the warp
roles are modelled as coroutines with the kernel's loop structure and its
slot / parity arithmetic (code ring of 3, K-block ring of 8, a ring of 4
accumulators each holding the partial sum of up to 8 K-blocks; the MMA warp
takes K-blocks in pairs; the two dequantising warps of each tensor-memory lane
quarter take the even and the odd K-blocks, counted over the whole launch so
that every K slot has one writer per quarter; a K slot's barrier counts the
four A writers and the B producer, whose copy lands on it), barriers with the PTX
test_wait / try_wait.parity semantics and the kernel's arrival counts, and TMA
landings and MMA commits completing in random order.  Every configuration
must finish without a stuck wait, every MMA must find the A and B blocks of
its own (unit, K-block) in its slot, and the epilogue must read every partial
sum of its own (unit, span) from its accumulator - i.e. no slot or
accumulator is overwritten while still in use."""
import itertools
import random

import pytest


class Bar:
    def __init__(s, count): s.count = count; s.pending = count; s.phase = 0; s.tx = 0
    def arrive(s, n=1):
        s.pending -= n
        s._maybe()
    def expect_tx(s, b): s.tx += b; s.arrive()
    def complete_tx(s, b): s.tx -= b; s._maybe()
    def _maybe(s):
        if s.pending == 0 and s.tx == 0:
            s.phase += 1; s.pending = s.count
    def done(s, parity):  # try_wait.parity semantics
        return (s.phase & 1) != parity

def sim(n_units, ng, kCS=3, kKS=8, D=4, SPAN=8, PAIR=2, seed=0, stage_parity=False):
    rnd = random.Random(seed)
    nst = (ng + 7) // 8
    full_c = [Bar(1) for _ in range(kCS)]; empty_c = [Bar(8) for _ in range(kCS)]
    # full_a: 4 dequantising warps + the B producer's expect_tx (B's bytes land on the same barrier)
    full_a = [Bar(5) for _ in range(kKS)]; empty_k = [Bar(1) for _ in range(kKS)]
    dfull = [Bar(1) for _ in range(D)]; dempty = [Bar(4) for _ in range(D)]
    smem_c = [None]*kCS; smem_a = [[None]*4 for _ in range(kKS)]; smem_b = [None]*kKS; tmem = [None]*D
    inflight = []  # (callback) async completions (TMA, MMA commit)
    log = {"mma": [], "epi": []}
    def producer_codes():
        cc = 0
        for u in range(n_units):
            for st in range(nst):
                slot = cc % kCS
                while not empty_c[slot].done(((cc // kCS) & 1) ^ 1): yield
                full_c[slot].expect_tx(100)
                tag = (u, st)
                def land(slot=slot, tag=tag):
                    smem_c[slot] = tag; full_c[slot].complete_tx(100)
                inflight.append(land)
                cc += 1
    def producer_b():
        kc = 0
        for u in range(n_units):
            for kb in range(ng):
                slot = kc % kKS
                while not empty_k[slot].done(((kc // kKS) & 1) ^ 1): yield
                full_a[slot].expect_tx(7)
                tag = (u, kb)
                def land(slot=slot, tag=tag):
                    smem_b[slot] = tag; full_a[slot].complete_tx(7)
                inflight.append(land)
                kc += 1
    def mma():
        kc = 0; pc = 0
        for u in range(n_units):
            for kb0 in range(0, ng, SPAN):
                d = pc % D
                while not dempty[d].done(((pc // D) & 1) ^ 1): yield
                tmem[d] = (u, kb0)
                kb1 = min(ng, kb0 + SPAN)
                kb = kb0
                while kb < kb1:
                    nkb = min(PAIR, kb1 - kb)
                    for i in range(nkb):
                        slot = (kc + i) % kKS; par = ((kc + i) // kKS) & 1
                        while not full_a[slot].done(par): yield
                    for i in range(nkb):
                        slot = (kc + i) % kKS
                        assert smem_a[slot] == [(u, kb + i)] * 4, (smem_a[slot], u, kb + i)
                        assert smem_b[slot] == (u, kb + i), (smem_b[slot], u, kb + i)
                        log["mma"].append((u, kb + i, d))
                        inflight.append(lambda slot=slot: empty_k[slot].arrive())
                    kb += nkb; kc += nkb
                inflight.append(lambda d=d: dfull[d].arrive())
                pc += 1
    def epi(w):
        pc = 0
        for u in range(n_units):
            for kb0 in range(0, ng, SPAN):
                d = pc % D
                while not dfull[d].done((pc // D) & 1): yield
                assert tmem[d] == (u, kb0), (tmem[d], u, kb0)
                if w == 0: log["epi"].append((u, kb0, d))
                dempty[d].arrive()
                pc += 1
    def deq(w):
        cc = 0; kc = 0
        for u in range(n_units):
            for st in range(nst):
                cs = cc % kCS
                while not full_c[cs].done((cc // kCS) & 1): yield
                assert smem_c[cs] == (u, st)
                gcount = min(8, ng - 8 * st)
                j0 = (w // 4) if stage_parity else (w // 4) ^ (kc & 1)  # kernel: kj % 2 == w // 4
                for j in range(j0, gcount, 2):
                    kj = kc + j; ks = kj % kKS
                    while not empty_k[ks].done(((kj // kKS) & 1) ^ 1): yield
                    smem_a[ks][w % 4] = (u, 8 * st + j)
                    full_a[ks].arrive()
                kc += gcount
                empty_c[cs].arrive()
                cc += 1
    roles = [producer_codes(), producer_b(), mma()] + [epi(i) for i in range(4)] + [deq(i) for i in range(8)]
    alive = list(roles); idle = 0
    while alive or inflight:
        progressed = False
        if inflight and rnd.random() < 0.5:
            inflight.pop(rnd.randrange(len(inflight)))(); progressed = True
        order = list(alive); rnd.shuffle(order)
        for r in order:
            try: next(r)
            except StopIteration: alive.remove(r); progressed = True
        if not alive and not inflight: break
        idle = 0 if progressed else idle + 1
        if idle > 2000 and not inflight: return False, log
    assert len(log["mma"]) == n_units * ng and len(log["epi"]) == n_units * ((ng + SPAN - 1) // SPAN)
    return True, log


@pytest.mark.parametrize("n_units", [0, 1, 2, 3, 5, 9])
@pytest.mark.parametrize("ng", [1, 2, 5, 8, 9, 16, 17, 64])
def test_protocol_completes_and_never_overwrites_live_slots(n_units, ng):
    for seed in range(3):
        for span in (4, 8):
            ok, _ = sim(n_units, ng, SPAN=span, seed=seed)
            assert ok, (n_units, ng, span, seed)


def test_model_catches_stage_relative_parity_with_odd_group_counts():
    # Splitting each stage's K-blocks by their index inside the stage lets one
    # warp of a quarter run a whole ring lap ahead when a unit has an odd
    # number of groups, so a slot parity aliases; the model must see it.
    bad = 0
    for ng in (5, 9, 17):
        for seed in range(6):
            try:
                ok, _ = sim(7, ng, seed=seed, stage_parity=True)
            except AssertionError:
                ok = False
            bad += not ok
    assert bad > 0
