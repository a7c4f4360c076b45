"""The logits kernel's and the backward GEMM's work orders, replayed on the CPU.

``unit_coords`` in ``csrc/rlk_logits.cu`` maps a work unit to (W tile, token
unit) in bands of 32 token tiles, vocabulary-major inside a band; the GEMM's
``decode`` in ``csrc/rlk_gemm.cu`` takes N tiles in bands when ``n_band`` is
set.  Each must visit every tile exactly once (a skipped or repeated tile
would leave logits unreduced or reduce them twice), and the bands must come
in order with every tile of a band before the next.
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


@pytest.mark.parametrize("pair", [False, True])
def test_logits_units_cover_every_tile_once_band_by_band(pair):
    band_mu = 16 if pair else 32
    for num_n in (1, 2, 3, 7, 594):
        for num_m in list(range(1, 70)) + [127, 128, 129]:
            num_mu = (num_m + 1) // 2 if pair else num_m
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
