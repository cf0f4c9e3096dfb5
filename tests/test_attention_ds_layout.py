"""Host-side model of the stored-dS attention backward's block layout (no GPU).

The key-side kernel writes one 128 x 128 dS block per (query tile, key tile,
head) that it visits, at slot (qt ktc + qt - kt) n_heads + h; the query-side
kernel reads the blocks of key tiles floor(seq_start / 128) .. qt.  Both rest on
the row metadata rule (a token continues the token before it, else it starts
a sequence; a position >= the bound is a range error and a one-token
sequence; padding rows are one-row sequences; a sequence never starts before
its adapter's padded segment) and on sequence starts not decreasing along the
padded rows.  This test rebuilds that rule and the two kernels' index rules
in plain Python over random layouts and checks, for every layout:
  * every block the query side reads is one the key side writes;
  * every slot lies inside the allocated [max_tiles x ktc x n_heads] blocks,
    with ktc = ceil((S - 1) / 128) + 1 for the sequence bound S;
  * the blocks read cover every causal (query, key) pair of the query tile,
    and the query tiles the key side visits cover every query that sees the
    key tile;
  * sequences longer than S leave range errors, never an out-of-range slot.
"""
import numpy as np
import pytest

TB = 128


def padded_layout(lengths, adapters, n_ad, S):
    """Rows in padded adapter order with the row metadata rule: returns
    (seq_start per padded row, number of range errors, padded row count)."""
    pos = np.concatenate([np.arange(L) for L in lengths]).astype(np.int64)
    ad = np.concatenate([np.full(L, a) for L, a in zip(lengths, adapters)]).astype(np.int64)
    n = len(pos)
    order = np.argsort(ad, kind="stable")
    counts = np.bincount(ad, minlength=n_ad)
    pad_off = np.concatenate([[0], np.cumsum((counts + TB - 1) // TB * TB)])
    P = int(pad_off[-1])
    seq_start = np.arange(P, dtype=np.int64)          # padding rows: one-row sequences
    errors = 0
    nxt = pad_off[:-1].copy()
    for t in order:
        a = ad[t]
        p = int(nxt[a])
        nxt[a] += 1
        q = int(pos[t])
        ok = 0 <= q < S
        if ok and q > 0:
            ok = t > 0 and pos[t - 1] == q - 1 and ad[t - 1] == a
        if ok:
            seq_start[p] = max(p - q, int(pad_off[a]))
        else:
            errors += 1
    assert n == counts.sum()
    return seq_start, errors, P


def check_layout(seq_start, P, S, n_heads):
    mt = P // TB
    ktc = -(-(S - 1) // TB) + 1
    cap = mt * ktc * n_heads
    assert np.all(np.diff(seq_start) >= 0), "sequence starts must not decrease along the rows"
    written = set()
    for kt in range(mt):                               # key side: item (kt, head group)
        nqt = 0
        while kt + nqt < mt and seq_start[(kt + nqt) * TB] <= kt * TB + TB - 1:
            nqt += 1
        assert nqt >= 1                                # its own tile
        for n in range(nqt):
            qt = kt + n
            assert qt - kt < ktc, (qt, kt, ktc)        # the kernel's range guard never fires
            for h in range(n_heads):
                slot = (qt * ktc + (qt - kt)) * n_heads + h
                assert 0 <= slot < cap
            written.add((qt, kt))
        # every query that sees a key of this tile lies in a visited query tile
        for j in range(kt * TB, kt * TB + TB):
            later = np.arange(j, P)
            sees = later[seq_start[later] <= j]
            assert sees.size == 0 or sees.max() // TB < kt + nqt
    for qt in range(mt):                               # query side: item (qt, head)
        kt0 = seq_start[qt * TB] // TB
        assert qt - kt0 < ktc                          # no clamp
        for kt in range(kt0, qt + 1):
            assert (qt, kt) in written, (qt, kt)
        rows = np.arange(qt * TB, qt * TB + TB)
        assert np.all(seq_start[rows] >= kt0 * TB)     # the read blocks cover every causal key
    return len(written), cap


@pytest.mark.parametrize("seed,S,n_ad,n_seq,hi", [
    (0, 300, 3, 12, 300),        # the small transformer workload's bound, all sequences within it
    (1, 300, 3, 12, 420),        # some sequences past the bound: range errors
    (2, 129, 5, 30, 200),        # a bound just past one tile
    (3, 1, 2, 40, 3),            # every sequence one token long (ktc = 1)
    (4, 2048, 4, 10, 2048),      # the benchmark's bound
    (5, 2048, 32, 24, 2600),     # many adapters, over-long sequences
])
def test_block_layout_invariants(seed, S, n_ad, n_seq, hi):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, hi + 1, n_seq)
    adapters = rng.integers(0, n_ad, n_seq)
    seq_start, errors, P = padded_layout(lengths, adapters, n_ad, S)
    n_blocks, cap = check_layout(seq_start, P, S, n_heads=4)
    assert n_blocks <= cap // 4
    over = int(np.maximum(lengths - S, 0).sum())
    assert errors == over                              # exactly the positions >= S


def test_capacity_formula_matches_worst_case():
    """A single sequence of exactly S tokens that starts mid-tile needs
    ceil((S - 1) / 128) + 1 key tiles for its last query tile."""
    for S in (1, 2, 127, 128, 129, 255, 256, 257, 2048):
        for lead in (0, 1, 64, 127):
            lengths = [lead, S] if lead else [S]
            seq_start, errors, P = padded_layout(lengths, [0] * len(lengths), 1, max(S, lead + 1))
            assert errors == 0
            ktc = -(-(S - 1) // TB) + 1
            last = (lead + S - 1) // TB
            kt0 = seq_start[last * TB] // TB
            assert last - kt0 + 1 <= ktc
