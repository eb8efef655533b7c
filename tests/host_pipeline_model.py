"""A model of attn_fwd_host's stream and event protocol, run under random
stream progress on the CPU.

attn_fwd_host (the forward on host-resident tensors) cuts a problem into
chunks of heads and pipelines them over a ring of device slots in the caller's
workspace with two internal streams per device, shared by every call on that
device:

* it records `start` on the caller's stream and makes both copy streams wait
  for it (everything starts after the caller's earlier work);
* per chunk c in slot c mod slots: the copy-in stream waits for the slot's
  `drained` event (for c >= slots), copies the inputs in and records `filled`;
  the caller's stream waits for `filled`, runs the kernel and records
  `computed`; the copy-out stream waits for `computed`, copies O and lse out
  and records `drained`;
* at the end it records `end` on the copy-out stream and `start` on the
  copy-in stream, and the caller's stream waits for both, so the caller's
  later work sees every copy of the call finished.

CUDA's rules, as modelled: operations on one stream run in order; recording an
event captures the work enqueued on that stream so far; a wait enqueued on a
stream waits for the event's most recent record at the time of the wait call
(none: no wait).  The host enqueues each call whole (the per-device mutex).
The checks: a slot is refilled only after the chunk it held was copied out, the
kernel reads the chunk that was copied in, the copy-out reads the chunk the
kernel wrote, and work the caller enqueues after a call finds every output of
that call copied back and none of its inputs still being read.
"""

from __future__ import annotations

import random


class PipelineError(AssertionError):
    pass


class Event:
    """A CUDA event: each record is a version; a wait refers to the version
    current when the wait was enqueued and is satisfied by that record's
    completion only (a later record on another stream does not count)."""

    def __init__(self, name):
        self.name, self.recorded, self.done = name, 0, set()


class Device:
    """One device: its two copy streams and events, plus the caller streams."""

    def __init__(self, slots=3, seed=0, mutant=None):
        self.slots, self.mutant = slots, mutant
        self.rnd = random.Random(seed)
        self.streams = {"in": [], "out": []}
        self.ev = {n: Event(n) for n in ("start", "end")}
        for s in range(slots):
            for n in ("filled", "computed", "drained"):
                self.ev[f"{n}{s}"] = Event(f"{n}{s}")
        self.slot_state = {}          # (workspace, slot) -> (stage, call, chunk)
        self.outputs = {}             # (call, chunk) -> copied back
        self.inputs_busy = {}         # call -> chunks whose inputs are still to be copied in
        self.call_chunks = {}

    # ------------------------------------------------------------ enqueueing
    def _push(self, stream, op):
        self.streams.setdefault(stream, []).append(op)

    def record(self, stream, name):
        e = self.ev[name]
        e.recorded += 1
        self._push(stream, ("record", e, e.recorded))

    def wait(self, stream, name):
        e = self.ev[name]
        if e.recorded:
            self._push(stream, ("wait", e, e.recorded))

    def call(self, call_id, stream, workspace, n_chunks, fail_at=None, copy_fails=False):
        """attn_fwd_host as enqueued by the host, in the library's order.
        `fail_at`: that chunk's kernel launch fails after its copy-in was
        enqueued (or, with `copy_fails`, one of its later input copies fails
        to enqueue, so no event follows the copy already in flight) and the
        call stops there, returning the error."""
        S = self.slots if n_chunks >= self.slots else n_chunks
        last = n_chunks if fail_at is None else fail_at + 1
        self.call_chunks[call_id] = n_chunks if fail_at is None else fail_at
        self.inputs_busy[call_id] = set(range(last))
        self.record(stream, "start")
        self.wait("in", "start")
        self.wait("out", "start")
        for c in range(n_chunks):
            slot = c % S
            if c >= S and self.mutant != "no_drained_wait":
                self.wait("in", f"drained{slot}")
            # a chunk whose kernel launch fails is copied in and never read
            self._push("in", ("copy_in", call_id, c, (workspace, slot), c == fail_at))
            if c == fail_at and copy_fails:
                break
            self.record("in", f"filled{slot}")
            self.wait(stream, f"filled{slot}")
            if c == fail_at:
                break
            self._push(stream, ("kernel", call_id, c, (workspace, slot)))
            self.record(stream, f"computed{slot}")
            self.wait("out", f"computed{slot}")
            self._push("out", ("copy_out", call_id, c, (workspace, slot)))
            self.record("out", f"drained{slot}")
        self.record("out", "end")
        self.wait(stream, "end")
        if self.mutant != "no_copy_in_tail":
            self.record("in", "start")
            self.wait(stream, "start")

    def user_work(self, call_id, stream):
        """Work the caller enqueues after the call: reads the outputs, may
        overwrite the inputs."""
        self._push(stream, ("user", call_id))

    # ------------------------------------------------------------- execution
    def _ready(self, op):
        return op[0] != "wait" or op[2] in op[1].done

    def _execute(self, op):
        kind = op[0]
        if kind == "record":
            op[1].done.add(op[2])
        elif kind == "wait":
            pass
        elif kind == "copy_in":
            _, call_id, c, key, abandoned = op
            st = self.slot_state.get(key)
            if st is not None and st[0] not in ("drained", "abandoned"):
                raise PipelineError(f"slot {key} refilled with chunk {c} of call {call_id} while "
                                    f"chunk {st[2]} of call {st[1]} is at stage {st[0]}")
            self.slot_state[key] = ("abandoned" if abandoned else "in", call_id, c)
            self.inputs_busy[call_id].discard(c)
        elif kind == "kernel":
            _, call_id, c, key = op
            if self.slot_state.get(key) != ("in", call_id, c):
                raise PipelineError(f"kernel of chunk {c} of call {call_id} found {self.slot_state.get(key)}")
            self.slot_state[key] = ("computed", call_id, c)
        elif kind == "copy_out":
            _, call_id, c, key = op
            if self.slot_state.get(key) != ("computed", call_id, c):
                raise PipelineError(f"copy-out of chunk {c} of call {call_id} found {self.slot_state.get(key)}")
            self.slot_state[key] = ("drained", call_id, c)
            self.outputs[(call_id, c)] = True
        elif kind == "user":
            call_id = op[1]
            missing = [c for c in range(self.call_chunks[call_id]) if not self.outputs.get((call_id, c))]
            if missing or self.inputs_busy[call_id]:
                raise PipelineError(f"work after call {call_id} ran with chunks {missing} not copied "
                                    f"out or chunks {sorted(self.inputs_busy[call_id])} still "
                                    f"being copied in")

    def run(self, max_steps=100000):
        for _ in range(max_steps):
            ready = [s for s, q in self.streams.items() if q and self._ready(q[0])]
            if not ready:
                if any(self.streams.values()):
                    raise PipelineError("streams wait forever: " + ", ".join(
                        s for s, q in self.streams.items() if q))
                return
            s = self.rnd.choice(ready)
            self._execute(self.streams[s].pop(0))
        raise PipelineError("no end within the step budget")
