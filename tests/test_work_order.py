"""The logits kernel's and the backward GEMM's work orders, replayed on the CPU.

``unit_coords`` in ``csrc/rlk_logits.cu`` maps a work unit to (W tile, token
tile) in bands of 32 token tiles, vocabulary-major inside a band; the GEMM's
``decode`` in ``csrc/rlk_gemm.cu`` takes N tiles in bands when ``n_band`` is
set.  Each must visit every tile exactly once (a skipped or repeated tile
would leave logits unreduced or reduce them twice), and the bands must come
in order with every tile of a band before the next.  The materialised-logits
kernel (``csrc/rlk_logits_mat.cu``) walks each warp's (row, slice) tasks by a
fixed (rows, slices) step; together the warps must take every slice of every
active row exactly once and no slice of an inactive row.
"""
import pytest


def unit_coords(unit, num_n, num_mu, band_mu):
    full = band_mu * num_n
    band = unit // full
    first_mu = band * band_mu
    mus = min(band_mu, num_mu - first_mu)
    within = unit - band * full
    n_blk = within // mus
    return n_blk, first_mu + (within - n_blk * mus)


def gemm_decode(r, num_m, num_n, n_band):
    n_band = n_band if 0 < n_band < num_n else num_n
    full = num_m * n_band
    band = r // full
    first_n = band * n_band
    nb = min(n_band, num_n - first_n)
    within = r - band * full
    m_blk = within // nb
    return m_blk, first_n + (within - m_blk * nb)


def test_logits_units_cover_every_tile_once_band_by_band():
    band_mu = 32
    for num_n in (1, 2, 3, 7, 594):
        for num_m in list(range(1, 70)) + [127, 128, 129]:
            num_mu = num_m
            seq = [unit_coords(u, num_n, num_mu, band_mu) for u in range(num_mu * num_n)]
            assert sorted(seq) == [(n, m) for n in range(num_n) for m in range(num_mu)]
            bands = [m // band_mu for _, m in seq]
            assert bands == sorted(bands)  # bands in order, each finished before the next
            if num_mu <= band_mu:  # one band: the plain vocabulary-major order
                assert seq == [(u // num_mu, u % num_mu) for u in range(num_mu * num_n)]


def test_gemm_units_cover_every_tile_once_band_by_band():
    for num_m in (1, 3, 8, 1187):
        for num_n in (1, 2, 5, 16, 17):
            for n_band in (0, 1, 3, 8, 16, 40):
                seq = [gemm_decode(r, num_m, num_n, n_band) for r in range(num_m * num_n)]
                assert sorted(seq) == [(m, n) for m in range(num_m) for n in range(num_n)]
                nb = n_band if 0 < n_band < num_n else num_n
                bands = [n // nb for _, n in seq]
                assert bands == sorted(bands)


def mat_walk(first, T, slices_per_row, stride, active):
    """One warp's (row, slice) tasks, stepped as the kernel steps them."""
    step_t, step_s = stride // slices_per_row, stride % slices_per_row

    def advance(t, s):
        t, s = t + step_t, s + step_s
        if s >= slices_per_row:
            s, t = s - slices_per_row, t + 1
        return t, s

    def skip_inactive(t, s):
        while t < T and active is not None and not active[t]:
            t, s = advance(t, s)
        return t, s

    t, s = skip_inactive(first // slices_per_row, first % slices_per_row)
    out = []
    while t < T:
        out.append((t, s))
        t, s = skip_inactive(*advance(t, s))
    return out


@pytest.mark.parametrize("masked", [False, True])
def test_mat_walk_takes_every_active_slice_once(masked):
    warps_per_cta = 4
    for T in (1, 2, 5, 37, 300):
        active = [(t * 7 + 3) % 5 != 0 for t in range(T)] if masked else None
        for slices_per_row in (1, 2, 3, 38, 75):
            n_tasks = T * slices_per_row
            for ctas in (1, 3, 152, 456, 760):
                blocks = min(ctas, (n_tasks + warps_per_cta - 1) // warps_per_cta)
                stride = blocks * warps_per_cta
                seen = []
                for first in range(stride):
                    walk = mat_walk(first, T, slices_per_row, stride, active)
                    # row-major task order, every stride-th task from `first`
                    tasks = [t * slices_per_row + s for t, s in walk]
                    assert all(b - a >= stride and (b - first) % stride == 0
                               for a, b in zip(tasks, tasks[1:]))
                    seen += walk
                want = [(t, s) for t in range(T) for s in range(slices_per_row)
                        if active is None or active[t]]
                assert sorted(seen) == want
