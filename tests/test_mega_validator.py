"""CPU checks of the megakernel's host queue validator (page
"Kernel-Mega-PDL", section 4: an instruction may wait only on events of
earlier instructions in the global order, whose signals reach the awaited
count, so the persistent grid cannot deadlock).  The validator runs on a
host array of 128-byte instructions through dl_test_validate_mega_queues;
no device is touched."""
import numpy as np
import pytest

import pdl_persistent_megakernel_gb300 as dl

NOOP = 0xFFFFFFFF
OK, INVALID_ARG, PLAN_INVALID = 0, 1, 6


def instr(op, cta=0, waits=(), signals=((None, 1),)):
    """One instruction as 32 uint32: op_row, cta, n_wait, n_signal,
    wait_event[4], wait_value[4], signal_event[0:2], signal_inc[0:2],
    signal_event[2:4], signal_inc[2:4], pad."""
    w = np.zeros(32, dtype=np.uint32)
    w[0], w[1] = op, cta
    w[2], w[3] = len(waits), len(signals)
    for k, (e, v) in enumerate(waits):
        w[4 + k], w[8 + k] = e, v
    for k, (e, inc) in enumerate(signals):
        base = 12 if k < 2 else 14
        w[base + k], w[base + 2 + k] = (op if e is None else e), inc
    return w


def noop():
    w = np.zeros(32, dtype=np.uint32)
    w[0] = NOOP
    return w


def chain_queues(n_ops, workers):
    """The plan builder's shape: op k's share c on worker c, each share
    waiting for all of op k - 1's shares, then a NoOp per queue."""
    q = np.zeros((workers, n_ops + 1, 32), dtype=np.uint32)
    for c in range(workers):
        for k in range(n_ops):
            waits = ((k - 1, workers),) if k > 0 else ()
            q[c, k] = instr(k, c, waits)
        q[c, n_ops] = noop()
    return q


def validate(q, n_events):
    q = np.ascontiguousarray(q, dtype=np.uint32)
    L = dl.lib()
    return L.dl_test_validate_mega_queues(q.ctypes.data, q.shape[0], q.shape[1], n_events)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    try:
        dl.lib()
    except (RuntimeError, FileNotFoundError, OSError) as e:  # no nvcc here
        pytest.skip(f"cannot build: {e}")


def test_plan_shaped_queues_pass():
    assert validate(chain_queues(7, 4), 7) == OK
    assert validate(chain_queues(1, 1), 1) == OK


def test_wait_on_a_later_op_is_rejected():
    q = chain_queues(3, 2)
    q[0, 1] = instr(1, 0, waits=((2, 1),))      # op 1 waits on op 2's event
    assert validate(q, 3) == PLAN_INVALID
    assert b"later op" in dl.lib().dl_last_error()


def test_wait_on_its_own_event_is_rejected():
    q = chain_queues(3, 2)
    q[1, 2] = instr(2, 1, waits=((2, 1),))
    assert validate(q, 3) == PLAN_INVALID


def test_unreachable_threshold_is_rejected():
    q = chain_queues(3, 2)
    q[0, 2] = instr(2, 0, waits=((1, 3),))      # op 1 signals only twice
    assert validate(q, 3) == PLAN_INVALID
    assert b"threshold" in dl.lib().dl_last_error()
    q[0, 2] = instr(2, 0, waits=((1, 2),))      # exactly reachable
    assert validate(q, 3) == OK


def test_signal_increments_are_summed_over_queues():
    q = chain_queues(2, 2)
    q[0, 0] = instr(0, 0, signals=((0, 3),))
    q[1, 0] = instr(0, 1, signals=((0, 2),))
    q[0, 1] = instr(1, 0, waits=((0, 5),))
    q[1, 1] = instr(1, 1, waits=((0, 5),))
    assert validate(q, 2) == OK
    q[1, 1] = instr(1, 1, waits=((0, 6),))
    assert validate(q, 2) == PLAN_INVALID


def test_queue_out_of_order_is_rejected():
    q = chain_queues(3, 2)
    q[0, [1, 2]] = q[0, [2, 1]]                 # op 2 before op 1 on worker 0
    assert validate(q, 3) == PLAN_INVALID
    assert b"order" in dl.lib().dl_last_error()


def test_instruction_after_the_terminator_is_rejected():
    q = np.zeros((1, 3, 32), dtype=np.uint32)
    q[0, 0] = instr(0)
    q[0, 1] = noop()
    q[0, 2] = instr(1, waits=((0, 1),))
    assert validate(q, 2) == PLAN_INVALID
    assert b"terminator" in dl.lib().dl_last_error()


def test_queue_without_terminator_is_rejected():
    q = chain_queues(2, 2)[:, :2]               # NoOp column cut off
    assert validate(q, 2) == PLAN_INVALID


def test_malformed_counts_and_events_are_rejected():
    q = chain_queues(2, 1)
    bad = q.copy()
    bad[0, 1, 2] = 5                            # n_wait > 4
    assert validate(bad, 2) == PLAN_INVALID
    bad = q.copy()
    bad[0, 0, 3] = 5                            # n_signal > 4
    assert validate(bad, 2) == PLAN_INVALID
    bad = q.copy()
    bad[0, 0, 12] = 7                           # signal of an unknown event
    assert validate(bad, 2) == PLAN_INVALID


def test_empty_description_is_an_argument_error():
    L = dl.lib()
    assert L.dl_test_validate_mega_queues(None, 1, 1, 1) == INVALID_ARG
    q = chain_queues(1, 1)
    assert validate(q, 0) == INVALID_ARG


def test_per_head_events_signalled_by_an_earlier_op():
    """Events that are not an op's own (the per-head events of a QKV
    projection): a later op may wait on them once their signals, from any
    instruction of earlier ops and in any of the four signal slots, reach
    the threshold; waiting on one that the same or a later op signals is a
    deadlock."""
    workers = 2
    # op 0 signals its own event and head events 2 and 3 (slots 2 and 3)
    q = np.zeros((workers, 3, 32), dtype=np.uint32)
    q[0, 0] = instr(0, 0, (), ((None, 1), (2, 1), (3, 2)))
    q[1, 0] = instr(0, 1, (), ((None, 1), (2, 1), (3, 1), (4, 1)))
    q[0, 1] = instr(1, 0, ((2, 2), (3, 3)))
    q[1, 1] = instr(1, 1, ((4, 1),))
    q[:, 2] = noop()
    assert validate(q, 5) == OK
    bad = q.copy()
    bad[1, 1] = instr(1, 1, ((3, 4),))          # only 3 signalled
    assert validate(bad, 5) == PLAN_INVALID
    bad = q.copy()
    bad[0, 1] = instr(1, 0, ((2, 2),), ((None, 1), (4, 1)))   # op 1 signals 4 ...
    assert validate(bad, 5) == PLAN_INVALID     # ... which op 1 waits on
