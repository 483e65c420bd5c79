"""Algorithmic HBM bytes of each call, from the sizes and the window counts.

These are the bytes the method must move (what a perfect kernel reads and
writes once), the denominator of the roofline fraction: the checkpoint is
read every step (bf16 read copy on non-flush steps when present) and written
only on a flush; the current record is read once and appended to the ring;
past records contribute the fields later steps read (Mamba-2 x, B, dt;
Gated DeltaNet k, g and the record's cached correction e, dv fp32 -- the
method keeps e beside each record, so v and beta are not read back; Kimi
Delta Attention the same with g one fp32 per key channel); outputs
are written once; each cursor is read and written (16 + 16 bytes).
"""

CURSOR = 32


def mamba2_parts(H, P, N, G, out_bytes):
    tile32 = H * P * N * 4                              # fp32 checkpoint of one sequence
    rec = 2 * H * P * 2 + 2 * G * N * 2 + H * 4        # x, z, B, C, dt of one token
    past = H * P * 2 + G * N * 2 + H * 4               # x, B, dt of one window record
    y = H * P * out_bytes
    return tile32, rec, past, y


def read_copy_bytes(H, P, N, read_copy):
    """Bytes of one sequence's read copy: 2 per element (bf16, fp16), or 1 per
    element plus a 4-byte scale per row (fp8); 0 without a copy."""
    if not read_copy:
        return 0
    if read_copy == "f8":
        return H * P * N + 4 * H * P
    return 2 * H * P * N


def mamba2_step_bytes(H, P, N, G, L, counts, read_copy=False, out_bytes=2):
    """One AR step; counts = each sequence's window count before the step."""
    tile32, rec, past, y = mamba2_parts(H, P, N, G, out_bytes)
    rc = read_copy_bytes(H, P, N, read_copy)
    total = 0
    for c in counts:
        if c + 1 == L:  # flush: read fp32, write fp32 (+ the read copy); the record is folded, not stored
            total += 2 * tile32 + rc + rec
        else:
            total += (rc if read_copy else tile32) + 2 * rec
        total += c * past + y + CURSOR
    return total


def mamba2_conventional_bytes(H, P, N, G, batch, out_bytes=2):
    tile32, rec, past, y = mamba2_parts(H, P, N, G, out_bytes)
    return batch * (2 * tile32 + rec + y)


def mamba2_verify_bytes(H, P, N, G, L, K, counts, read_copy=False, out_bytes=2):
    """One verify + commit; counts = committed window counts before the verify."""
    tile32, rec, past, y = mamba2_parts(H, P, N, G, out_bytes)
    rc = read_copy_bytes(H, P, N, read_copy)
    total = 0
    for c in counts:
        fold = c + K > L
        if fold:
            total += 2 * tile32 + rc
        else:
            total += rc if read_copy else tile32
        total += 2 * K * rec + c * past + K * y + 2 * CURSOR + 4
    return total


def gdn_parts(H, DK, DV, out_bytes):
    tile = H * DV * DK * 4
    rec = H * (2 * DK * 2 + DV * 2 + 8)                # q, k, v, g, beta
    e = H * DV * 4                                     # a record's cached correction
    past = H * (DK * 2 + 4) + e                        # k, g, e
    o = H * DV * out_bytes
    return tile, rec, e, past, o


def gdn_step_bytes(H, DK, DV, L, counts, out_bytes=2):
    tile, rec, e, past, o = gdn_parts(H, DK, DV, out_bytes)
    total = 0
    for c in counts:
        if c + 1 == L:
            total += 2 * tile + rec
        else:
            total += tile + 2 * rec + e
        total += c * past + o + CURSOR
    return total


def gdn_verify_bytes(H, DK, DV, L, K, counts, out_bytes=2):
    """One verify + commit; counts = committed window counts before the verify."""
    tile, rec, e, past, o = gdn_parts(H, DK, DV, out_bytes)
    total = 0
    for c in counts:
        total += 2 * tile if c + K > L else tile
        total += K * (2 * rec + e) + c * past + K * o + 2 * CURSOR + 4
    return total


def gdn_conventional_bytes(H, DK, DV, batch, out_bytes=2):
    tile, rec, e, past, o = gdn_parts(H, DK, DV, out_bytes)
    return batch * (2 * tile + rec + o)


def kda_parts(H, DK, DV, out_bytes):
    tile = H * DV * DK * 4
    rec = H * (2 * DK * 2 + DV * 2 + DK * 4 + 4)       # q, k, v, g (per key channel), beta
    e = H * DV * 4                                     # a record's cached correction
    past = H * (DK * 2 + DK * 4) + e                   # k, g, e
    o = H * DV * out_bytes
    return tile, rec, e, past, o


def kda_step_bytes(H, DK, DV, L, counts, out_bytes=2):
    tile, rec, e, past, o = kda_parts(H, DK, DV, out_bytes)
    total = 0
    for c in counts:
        if c + 1 == L:
            total += 2 * tile + rec
        else:
            total += tile + 2 * rec + e
        total += c * past + o + CURSOR
    return total


def kda_verify_bytes(H, DK, DV, L, K, counts, out_bytes=2):
    """One verify + commit; counts = committed window counts before the verify."""
    tile, rec, e, past, o = kda_parts(H, DK, DV, out_bytes)
    total = 0
    for c in counts:
        total += 2 * tile if c + K > L else tile
        total += K * (2 * rec + e) + c * past + K * o + 2 * CURSOR + 4
    return total


def kda_conventional_bytes(H, DK, DV, batch, out_bytes=2):
    tile, rec, e, past, o = kda_parts(H, DK, DV, out_bytes)
    return batch * (2 * tile + rec + o)
