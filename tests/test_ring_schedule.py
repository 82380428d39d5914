"""Host-side model of the piece schedule of the warp-specialised tensor-core
kernel (tiled_mma_ring_kernel.cuh), run under random interleavings of its three
actors: the copy engine, the producer (TMA issue and transposition) and the
consumers (MMAs).  Checks what the kernel's correctness rests on:

  - the copy cursor emits exactly the pieces the unit loop consumes, and their
    count is the closed form the kernel uses;
  - every parity wait is for the barrier's current or previous phase (an
    mbarrier parity wait cannot tell phase c from phase c + 2);
  - each piece is released exactly once (the last piece at most once);
  - a unit reads, from its two ring slots, the input pieces of its own column
    and band, and no slot is overwritten while a unit still reads it;
  - no interleaving deadlocks.
"""
from __future__ import annotations

import random

import pytest

NSLOT, NSTAGE = 3, 2  # ring slots, staging slots


class Bar:
    """An mbarrier: completes a phase after `count` arrivals."""

    def __init__(self, count=1):
        self.count = self.pending = count
        self.phase = 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def ready(self, c):
        """Waiting for phase c: legal only while the barrier is in phase c or c + 1."""
        assert c <= self.phase <= c + 1, f"parity wait for phase {c} at phase {self.phase}"
        return self.phase == c + 1


def cta_range(units, grid, b):
    return units * b // grid, units * (b + 1) // grid


def piece_list(u_begin, u_end, tiles_h):
    """The copy cursor of the kernel's producer: (column, piece row) per piece."""
    out = []
    for k, u in enumerate(range(u_begin, u_end)):
        col, band = divmod(u, tiles_h)
        if k == 0 or band == 0:
            out.append((col, band))
        out.append((col, band + 1))
    return out


def n_pieces(u_begin, u_end, tiles_h):
    """The kernel's closed form."""
    if u_end <= u_begin:
        return 0
    return (u_end - u_begin) + 1 + ((u_end - 1) // tiles_h - u_begin // tiles_h)


def run_cta(u_begin, u_end, tiles_h, rng, release_column_end=True):
    seq = piece_list(u_begin, u_end, tiles_h)
    npc = n_pieces(u_begin, u_end, tiles_h)
    assert len(seq) == npc
    sfull = [Bar() for _ in range(NSTAGE)]
    tfull = [Bar() for _ in range(NSLOT)]
    tempty = [Bar() for _ in range(NSLOT)]
    staging = [None] * NSTAGE
    ring = [None] * NSLOT
    readers = [0] * NSLOT
    inflight = []
    issued = [0]
    released = [0] * npc

    def issue():
        inflight.append(issued[0])
        issued[0] += 1

    def producer():
        for _ in range(min(NSTAGE, npc)):
            issue()
        for j in range(npc):
            slot, ss = j % NSLOT, j % NSTAGE
            if j >= NSLOT:
                while not tempty[slot].ready(j // NSLOT - 1):
                    yield
            while not sfull[ss].ready(j // NSTAGE):
                yield
            assert staging[ss] == j
            assert readers[slot] == 0, "ring slot overwritten while a unit reads it"
            ring[slot] = seq[j]
            yield
            tfull[slot].arrive()
            staging[ss] = None
            if issued[0] < npc:
                issue()
            yield

    def consumer():
        pc = 0
        for k, u in enumerate(range(u_begin, u_end)):
            col, band = divmod(u, tiles_h)
            fill = k == 0 or band == 0
            q = pc + 1 if fill else pc
            pc += 2 if fill else 1
            if fill:
                while not tfull[(q - 1) % NSLOT].ready((q - 1) // NSLOT):
                    yield
            while not tfull[q % NSLOT].ready(q // NSLOT):
                yield
            a, b = (q - 1) % NSLOT, q % NSLOT
            readers[a] += 1
            readers[b] += 1
            assert ring[a] == (col, band) and ring[b] == (col, band + 1)
            yield
            assert ring[a] == (col, band) and ring[b] == (col, band + 1)
            readers[a] -= 1
            readers[b] -= 1
            tempty[a].arrive()
            released[q - 1] += 1
            if band + 1 == tiles_h and release_column_end:
                tempty[b].arrive()
                released[q] += 1
            yield

    def copy_engine():
        while True:
            if inflight and rng.random() < 0.5:
                j = inflight.pop(0)
                ss = j % NSTAGE
                assert staging[ss] is None, "copy into a staging slot still in use"
                staging[ss] = j
                sfull[ss].arrive()
            yield

    actors = [producer(), consumer()]
    done = [False, False]
    engine = copy_engine()
    for _ in range(4000 * (npc + 1)):
        if all(done):
            break
        i = rng.randrange(3)
        if i == 2:
            next(engine)
        elif not done[i]:
            try:
                next(actors[i])
            except StopIteration:
                done[i] = True
    else:
        raise AssertionError("deadlock")
    assert all(r == 1 for r in released[:-1]) and released[-1] <= 1


@pytest.mark.parametrize("units,grid,tiles_h", [
    (2688, 152, 7),   # 128 images x 3 channel tiles of a 56x56 map
    (168, 152, 7),    # ranges of one or two units
    (960, 152, 5),    # ragged last band
    (64, 5, 1),       # columns of one band: every unit refills
    (300, 17, 2),
    (37, 3, 13),
    (9, 2, 9),
    (7, 7, 7),
])
def test_ring_schedule(units, grid, tiles_h):
    rng = random.Random(units * 131 + grid * 7 + tiles_h)
    for b in range(grid):
        u_begin, u_end = cta_range(units, grid, b)
        if u_end > u_begin:
            run_cta(u_begin, u_end, tiles_h, rng)


def test_piece_count_closed_form():
    for tiles_h in (1, 2, 3, 7, 13):
        for u_begin in range(0, 40):
            for u_end in range(u_begin, u_begin + 30):
                assert n_pieces(u_begin, u_end, tiles_h) == len(piece_list(u_begin, u_end, tiles_h))


def test_the_model_catches_a_missing_release():
    """Without the release of a column's last piece the producer waits for a
    ring-slot phase that never completes: the model must report a deadlock."""
    with pytest.raises(AssertionError, match="deadlock"):
        run_cta(0, 20, 3, random.Random(5), release_column_end=False)
