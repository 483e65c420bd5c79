"""Integer model of the per-sequence ring-buffer cursors (oracle; test-only).

Sources: "ReplaySSM Caches Inputs Instead of State...", section "How ReplaySSM
works" (append on non-flush steps; the L-th step folds the buffer and clears
it; drafts are appended instead of snapshotting state) and "ReplaySSM" (code
repository), introduction ("Cheap rollback": rejected inputs are discarded by
moving a buffer pointer). "ReplaySSM (a vLLM research fork)", section "Core
implementation files", names the commit and reset calls of the speculative
path. The exact buffer policy is not printed; the rules below are this
build's reading of it.

A cursor is four integers ``(start, count, pending, flags)``:

* ``start``   ring slot of the oldest record since the checkpoint, in [0, L);
* ``count``   committed records in the window, in [0, L];
* ``pending`` records appended by the last verify and not yet committed;
* ``flags``   bit 0 (``FOLDED``): that verify folded the committed window.

Rules (L = window length, K = records per verify):

* AR step: needs count < L and pending == 0. The record goes to slot
  (start + count) mod L. If count + 1 == L the step folds all L records
  (flush) and the cursor becomes (start, 0, 0, 0); else count += 1.
* Verify: needs count <= L, pending == 0, 1 <= K <= L. fold = count + K > L.
  Draft i goes to slot (start + count + i) mod L. Cursor becomes
  (start, count, K, FOLDED if fold else 0).
* Commit(kept): needs 0 <= kept <= pending. If FOLDED: start += count (mod L),
  count = 0. Then count += kept, pending = 0, flags = 0.
* Flush (standalone): needs pending == 0; folds the count records,
  start += count (mod L), count = 0.
* Reset: (0, 0, 0, 0).

A call whose precondition fails leaves that cursor unchanged and reports an
error for that sequence.
"""

FOLDED = 1


def valid_base(cur, L):
    start, count, pending, flags = cur
    return 0 <= start < L and 0 <= count <= L and pending >= 0


def ar_step(cur, L):
    """Returns (new_cursor, slot, flush, ok)."""
    start, count, pending, flags = cur
    if not (valid_base(cur, L) and count < L and pending == 0):
        return tuple(cur), None, False, False
    slot = (start + count) % L
    if count + 1 == L:
        return (start, 0, 0, 0), slot, True, True
    return (start, count + 1, 0, 0), slot, False, True


def verify(cur, K, L):
    """Returns (new_cursor, slots, fold, ok)."""
    start, count, pending, flags = cur
    if not (valid_base(cur, L) and pending == 0 and 1 <= K <= L):
        return tuple(cur), None, False, False
    fold = count + K > L
    slots = [(start + count + i) % L for i in range(K)]
    return (start, count, K, FOLDED if fold else 0), slots, fold, True


def commit(cur, kept, L):
    """Returns (new_cursor, ok)."""
    start, count, pending, flags = cur
    if not (valid_base(cur, L) and 0 <= kept <= pending):
        return tuple(cur), False
    if flags & FOLDED:
        start = (start + count) % L
        count = 0
    return (start, count + kept, 0, 0), True


def flush(cur, L):
    """Returns (new_cursor, folded_count, ok)."""
    start, count, pending, flags = cur
    if not (valid_base(cur, L) and pending == 0):
        return tuple(cur), 0, False
    return ((start + count) % L, 0, 0, 0), count, True


def reset(cur):
    return (0, 0, 0, 0)
