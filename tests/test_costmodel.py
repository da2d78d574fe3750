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


def test_data_stages_by_hand():
    # 8 ranks, int32, 16 channels, 512 KiB chunks: 1 KiB per rank is 256
    # elements, 16 per channel; the last loop's chunk is alignUp(2, 4) = 4
    # elements, so 4 of the 8 chunks hold data: 7 stages.
    assert cm.data_stages(256, 8, 16, 512 << 10, 4) == 7
    # 2 KiB: 32 per channel, chunks of 4: all 8 hold data: 15 stages.
    assert cm.data_stages(512, 8, 16, 512 << 10, 4) == 15
    # 8 bytes: 2 elements, one chunk of 4: 1 stage.
    assert cm.data_stages(2, 8, 16, 512 << 10, 4) == 1
    # a whole loop per channel: 2N - 1.
    assert cm.data_stages(1 << 26, 8, 16, 512 << 10, 4) == 15
    assert cm.data_stages(0, 8, 16, 512 << 10, 4) == 0


def test_fit_steps_recovers_parameters():
    truth = cm.StepParams(base_us=6.0, step_us=0.4, byte_us=3e-4)
    pts = []
    for n in (4, 8, 16):
        for b, parts, rings, g in ((1 << 10, 16, 16, 3), (1 << 16, 16, 16, 2 * n - 1),
                                   (1 << 24, 600, 152, 2 * n - 1), (1 << 28, 9000, 304, 2 * n - 1)):
            pts.append((b, n, parts, rings, g,
                        cm.predict_steps_us(truth, n, parts, rings, g, b)))
    got = cm.fit_steps(pts)
    assert math.isclose(got.base_us, truth.base_us, rel_tol=1e-6)
    assert math.isclose(got.step_us, truth.step_us, rel_tol=1e-6)
    assert math.isclose(got.byte_us, truth.byte_us, rel_tol=1e-6)
    assert max(abs(r) for r in cm.residuals_steps(got, pts)) < 1e-9


def test_step_formula_by_hand():
    # 2 passes of 15 stages, steps of 2^20 / (64 * 8) = 2048 bytes:
    # 5 + 2 * 15 * (0.5 + 2048 * 1e-4) = 26.144 us.
    p = cm.StepParams(base_us=5.0, step_us=0.5, byte_us=1e-4)
    assert math.isclose(cm.predict_steps_us(p, 8, 64, 32, 15, 1 << 20), 26.144)
