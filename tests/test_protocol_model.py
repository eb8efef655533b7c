"""The forward kernel's barrier protocol under random interleavings (CPU).

tests/protocol_model.py restates the synchronisation of attn_tc_kernel for
16-bit inputs, for e4m3 with V widened once per call and for e4m3 with V
widened on chip (the producer's K/V ring, one MMA issuer per query tile, the
score buffer the two tiles share, the softmax warps, the four V shares) and
checks, at every step of thousands of random schedules, that no mbarrier
parity wait is fooled, no buffer is read before it is written or overwritten
while still needed, and nothing deadlocks.  The planted mistakes below (a slot
released by one issuer only, a score MMA that does not wait for the other
tile's softmax, a softmax that overwrites P without waiting for the P V
reading it, a V share that does not wait for its fp16 buffer, the producer's
share lagging by half the ring) must each be caught.  The head-dimension-256
kernel (attn_tc256_kernel: one query tile, two score buffers with P written
over its scores, half-tile ring items, two V converters for e4m3) gets the
same treatment, with its two historical hazards planted: one P barrier for
both buffers, and an epilogue that waits on pv_done instead of o_done.  So do
the backward kernels: bwd_dkdv as built, and bwd_dq with its per-half dS
barriers kept one per step parity (the model shows that with one barrier per
half, as the kernel has them now, a warp lagging a whole half step behind the
others lets a faster warp's next-step arrival complete the phase: a parity
wait two phases behind, or dQ reading a dS half not yet written).

The abort path of the d <= 128 kernel is modelled too: at a random moment one
blocked wait runs out, every role leaves as the kernel's code does, and when
all roles are done (the CTA's exit) no TMA load and no MMA may still be in
flight.  That holds when the producer and the issuers drain at the end of
their roles whatever happened; as built they drain only when their own wait
failed, so a role that had already finished leaves its last loads or MMAs
undrained (tracked as an open item, like the dS barriers above).
"""

import pytest

from protocol_model import Kernel, Kernel256, KernelBwdDkdv, KernelBwdDq, ProtocolError

# ring depths the kernel uses: 5 slots (16-bit, d = 128), 6 (e4m3 K with
# fp16 V, d = 128), 8 (d = 64)
SLOTS = (5, 6, 8)
# key tiles of query tiles A and B: non-causal, causal (B one tile more),
# ragged (a tile with no key, or past the end of the queries), and a split-KV
# share; (0, 0) launches nothing
N_KV = [(1, 1), (2, 2), (5, 5), (9, 9), (1, 2), (3, 4), (7, 8), (0, 1), (2, 0), (3, 0),
        (0, 0), (2, 3)]


@pytest.mark.parametrize("slots", SLOTS)
@pytest.mark.parametrize("n_kv", N_KV, ids=lambda n: f"{n[0]}x{n[1]}")
def test_protocol_holds_under_random_schedules(n_kv, slots):
    for seed in range(60):
        Kernel(n_kv, slots, seed=1000 * slots + seed).run()


@pytest.mark.parametrize("n_kv", N_KV, ids=lambda n: f"{n[0]}x{n[1]}")
def test_on_chip_widening_protocol_holds_under_random_schedules(n_kv):
    # e4m3 with V widened on chip: 8 slots, K in even slots and V in odd ones
    for seed in range(60):
        Kernel(n_kv, 8, seed=seed, conv=True).run()


@pytest.mark.parametrize("mutant,conv", [("one_release_per_slot", False), ("no_s_free_wait", False),
                                         ("no_pv_wait", False), ("no_v16_empty_wait", True),
                                         ("lag_half_ring", True)])
def test_planted_protocol_mistakes_are_caught(mutant, conv):
    # (the producer's share lagging by half the ring deadlocks: the slot it
    # waits to refill is released only by its own share, which comes later)
    caught = 0
    for seed in range(200):
        for n_kv in [(3, 4), (5, 5)]:
            try:
                Kernel(n_kv, 8 if conv else 5, seed=seed, mutant=mutant, conv=conv).run()
            except ProtocolError:
                caught += 1
    assert caught > 0, f"{mutant} was never caught"


@pytest.mark.parametrize("e4m3", [False, True], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8, 17])
def test_d256_protocol_holds_under_random_schedules(n, e4m3):
    for seed in range(60):
        Kernel256(n, seed, e4m3=e4m3).run()


@pytest.mark.parametrize("mutant", ["one_p_barrier", "epilogue_on_pv_done"])
def test_d256_planted_mistakes_are_caught(mutant):
    caught = 0
    for seed in range(200):
        for e4m3 in (False, True):
            try:
                Kernel256(5, seed, e4m3=e4m3, mutant=mutant).run()
            except ProtocolError:
                caught += 1
    assert caught > 0, f"{mutant} was never caught"


@pytest.mark.parametrize("slots", [2, 5])          # the ring depths at d = 128 and 64
@pytest.mark.parametrize("steps", [1, 2, 3, 5, 9, 16])
def test_bwd_dkdv_protocol_holds_under_random_schedules(steps, slots):
    for seed in range(60):
        KernelBwdDkdv(steps, slots, seed).run()


@pytest.mark.parametrize("ks", [3, 4])              # K slots at d = 128 and 64; two V slots
@pytest.mark.parametrize("n", [1, 2, 3, 5, 9, 16])
def test_bwd_dq_protocol_with_per_parity_dS_barriers_holds(n, ks):
    for seed in range(60):
        KernelBwdDq(n, seed, ks=ks, robust=True).run()


def test_bwd_dq_with_one_dS_barrier_per_half_needs_bounded_warp_skew():
    # the form the kernel has today: some schedules with one warp a whole half
    # step behind break it (tracked as an open item; the form above is the fix)
    failures = 0
    for seed in range(150):
        try:
            KernelBwdDq(9, seed, robust=False).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


ABORT_N_KV = [(1, 1), (2, 2), (5, 5), (9, 9), (1, 2), (3, 4), (7, 8), (0, 1), (2, 0), (2, 3)]


@pytest.mark.parametrize("conv,slots", [(False, 5), (False, 6), (False, 8), (True, 8)],
                         ids=["16bit-5", "16bit-6", "16bit-8", "onchip-8"])
def test_abort_path_with_drains_at_every_role_end_leaves_nothing_in_flight(conv, slots):
    aborted = 0
    for n_kv in ABORT_N_KV:
        for seed in range(40):
            k = Kernel(n_kv, slots, seed, conv=conv, timeout_p=0.02, drain_always=True)
            k.run()
            aborted += k.abort
    assert aborted > 200        # most runs took the abort path somewhere


def test_abort_path_as_built_can_leave_work_in_flight():
    # a role that finished its loop before another role's wait ran out does not drain
    failures = 0
    for n_kv in ABORT_N_KV:
        for seed in range(40):
            try:
                Kernel(n_kv, 5, seed, timeout_p=0.02).run()
            except ProtocolError:
                failures += 1
    assert failures > 0
