"""The ring cost model (host logic, CPU): the pages' formula by hand, fitting
recovers known parameters, crossovers sit where the predictions meet."""
import math

import pytest

from ring_allreduce_virtual_gb300 import costmodel as cm


def test_formula_by_hand():
    # lat = 10 + 2*7*1 = 24 us; bw = 100 * 8 / 14 GB/s; 1 GB / bw = 17500 us.
    p = cm.ProtoParams(base_us=10.0, hop_us=1.0, bus_gbs=100.0)
    assert p.lat_us(8) == 24.0
    assert math.isclose(p.bw_gbs(8), 100.0 * 8 / 14)
    assert math.isclose(cm.predict_us(p, 1e9, 8), 24.0 + 17500.0)


def test_page_discounts():
    assert cm.PAGE_DISCOUNT == {"simple": 1.0, "ll": 0.5, "ll128": 0.9375}


def test_fit_recovers_parameters():
    truth = cm.ProtoParams(base_us=7.5, hop_us=0.8, bus_gbs=640.0)
    pts = [(b, n, cm.predict_us(truth, b, n)) for n in (4, 8, 16)
           for b in (1 << 10, 1 << 16, 1 << 20, 1 << 24, 1 << 28)]
    got = cm.fit(pts)
    assert math.isclose(got.base_us, truth.base_us, rel_tol=1e-6)
    assert math.isclose(got.hop_us, truth.hop_us, rel_tol=1e-6)
    assert math.isclose(got.bus_gbs, truth.bus_gbs, rel_tol=1e-6)
    assert max(abs(r) for r in cm.residuals(got, pts)) < 1e-9


def test_fit_one_ring_size_puts_latency_in_base():
    truth = cm.ProtoParams(base_us=5.0, hop_us=0.5, bus_gbs=300.0)
    pts = [(b, 8, cm.predict_us(truth, b, 8)) for b in (1 << 8, 1 << 14, 1 << 20, 1 << 26)]
    got = cm.fit(pts)
    assert got.hop_us == 0.0
    assert math.isclose(got.base_us, truth.lat_us(8), rel_tol=1e-6)
    assert math.isclose(got.bus_gbs, truth.bus_gbs, rel_tol=1e-6)


def test_crossover_is_where_times_meet():
    ll = cm.ProtoParams(base_us=4.0, hop_us=0.2, bus_gbs=250.0)
    simple = cm.ProtoParams(base_us=9.0, hop_us=0.6, bus_gbs=650.0)
    x = cm.crossover_bytes(ll, simple, 8)
    assert x is not None and x > 0
    assert math.isclose(cm.predict_us(ll, x, 8), cm.predict_us(simple, x, 8), rel_tol=1e-9)
    assert cm.predict_us(ll, x / 2, 8) < cm.predict_us(simple, x / 2, 8)
    assert cm.predict_us(ll, x * 2, 8) > cm.predict_us(simple, x * 2, 8)


def test_no_crossover_when_one_dominates():
    fast = cm.ProtoParams(base_us=1.0, hop_us=0.1, bus_gbs=900.0)
    slow = cm.ProtoParams(base_us=5.0, hop_us=0.5, bus_gbs=200.0)
    assert cm.crossover_bytes(fast, slow, 8) is None


def test_passes_model():
    assert cm.passes(0, 152) == 0 and cm.passes(1, 152) == 1
    assert cm.passes(152, 152) == 1 and cm.passes(153, 152) == 2
    truth = cm.PassParams(base_us=6.0, stage_us=0.7, bus_gbs=600.0)
    # 8 ranks: 15 stages per pass; 1 GB at 600 * 8 / 14 GB/s
    assert math.isclose(cm.predict_passes_us(truth, 8, 3, 1e9),
                        6.0 + 3 * 15 * 0.7 + 1e9 / (1000 * 600 * 8 / 14))
    pts = [(b, n, k, cm.predict_passes_us(truth, n, k, b)) for n in (4, 8, 16)
           for k, b in ((1, 1 << 10), (2, 1 << 20), (7, 1 << 24), (40, 1 << 28))]
    got = cm.fit_passes(pts)
    assert math.isclose(got.base_us, 6.0, rel_tol=1e-6)
    assert math.isclose(got.stage_us, 0.7, rel_tol=1e-6)
    assert math.isclose(got.bus_gbs, 600.0, rel_tol=1e-6)
    assert max(abs(r) for r in cm.residuals_passes(got, pts)) < 1e-9
