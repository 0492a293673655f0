"""The oracle's continuous-batching step on several host processes at once.

Test and baseline infrastructure, like the rest of this package: only the
CPU-baseline leg of bench.py runs it, to report how fast the plain fp64
oracle goes on all the host's cores. It adds no arithmetic of its own: each
process repeats ``block_hybrid.attend`` for every request of a sample and
``block_hybrid.commit`` for the committing ones.
"""

from __future__ import annotations

import time

from oracle import block_hybrid as ob


def one_step(t, states, commit) -> None:
    """One step of the sample: attend for every request, commit for the
    requests in ``commit`` (their new states are discarded, so every step
    does the same work)."""
    for b, (S, Z) in enumerate(states):
        ob.attend(t["q"][b], t["k"][b], t["v"][b], S, Z, t["W"], t["gate"], ob.MERGE_SHARED_NORM)
        if b in commit:
            ob.commit(S, Z, t["k"][b], t["v"][b], t["W"])


def timed_steps(args) -> tuple:
    """Runs steps until ``seconds`` have passed; returns (steps, seconds)."""
    t, states, commit, seconds = args
    one_step(t, states, commit)  # warm the process's caches
    t0 = time.perf_counter()
    reps = 0
    while True:
        one_step(t, states, commit)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return reps, el
