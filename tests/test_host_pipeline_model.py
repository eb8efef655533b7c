"""attn_fwd_host's stream and event protocol under random stream progress (CPU).

tests/host_pipeline_model.py restates the order in which attn_fwd_host
enqueues its copies, kernels, event records and waits on the caller's stream
and the device's two shared copy streams, with CUDA's event semantics, and
checks under thousands of random interleavings of the streams that no
workspace slot is refilled while the chunk it holds is still to be computed or
copied out, and that work the caller enqueues after a call sees all of that
call's copies finished: for one call, calls back to back on one stream, the
end-to-end benchmark's pattern (steps issued back to back on two caller
streams with a workspace each, sharing the copy streams), and calls that stop
early on an error.  Planted mistakes (no wait for a slot's copy-out before
refilling it, no copy-in tail at the end of a call) are caught.
"""

import pytest

from host_pipeline_model import Device, PipelineError

CHUNKS = [1, 2, 3, 4, 7]


def _scenario(kind, n_chunks, seed, mutant=None):
    d = Device(slots=3, seed=seed, mutant=mutant)
    if kind == "one":
        d.call(0, "A", "wsA", n_chunks)
        d.user_work(0, "A")
    elif kind == "same_stream":
        for i in range(3):
            d.call(i, "A", "wsA", n_chunks)
            d.user_work(i, "A")
    else:   # two caller streams, a workspace each, steps back to back, joined at the end
        for step in range(4):
            d.call(2 * step, "A", "wsA", n_chunks)
            d.call(2 * step + 1, "B", "wsB", n_chunks)
        for i in range(8):
            d.user_work(i, "A" if i % 2 == 0 else "B")
    d.run()


@pytest.mark.parametrize("kind", ["one", "same_stream", "two_streams"])
@pytest.mark.parametrize("n_chunks", CHUNKS)
def test_pipeline_protocol_holds(kind, n_chunks):
    for seed in range(60):
        _scenario(kind, n_chunks, seed)


@pytest.mark.parametrize("copy_fails", [False, True], ids=["launch_fails", "copy_fails"])
@pytest.mark.parametrize("n_chunks", [1, 2, 4, 7])
def test_a_call_that_stops_on_an_error_leaves_nothing_behind(n_chunks, copy_fails):
    # the next call reuses the same workspace and stream
    for fail_at in range(n_chunks):
        for seed in range(30):
            d = Device(slots=3, seed=seed)
            d.call(0, "A", "wsA", n_chunks, fail_at=fail_at, copy_fails=copy_fails)
            d.user_work(0, "A")
            d.call(1, "A", "wsA", n_chunks)
            d.user_work(1, "A")
            d.run()


def test_refilling_a_slot_without_waiting_for_its_copy_out_is_caught():
    caught = 0
    for seed in range(100):
        try:
            _scenario("one", 7, seed, mutant="no_drained_wait")
        except PipelineError:
            caught += 1
    assert caught > 0


def test_dropping_the_copy_in_tail_is_caught():
    # only a call whose input copy failed to enqueue relies on it
    caught = 0
    for seed in range(200):
        for fail_at in range(4):
            d = Device(slots=3, seed=seed, mutant="no_copy_in_tail")
            d.call(0, "A", "wsA", 4, fail_at=fail_at, copy_fails=True)
            d.user_work(0, "A")
            try:
                d.run()
            except PipelineError:
                caught += 1
    assert caught > 0
