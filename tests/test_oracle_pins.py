"""The CPU oracle against its pins (library routines, closed forms,
invariants, special cases).  CPU only."""
import pytest

import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.FFN_PINS, ids=lambda f: f.__name__)
def test_ffn_pin(pin):
    pin()


@pytest.mark.parametrize("pin", pins.FORMAT_PINS, ids=lambda f: f.__name__)
def test_format_pin(pin):
    pin()


@pytest.mark.parametrize("case", pins.ALIGN_CASES, ids=lambda c: "T%d_K%d_E%d_bm%d_%s" % c)
def test_align_vs_stable_argsort(case):
    pins.pin_align_vs_stable_argsort(*case)


def test_align_invariants():
    pins.pin_align_invariants()


def test_align_rejects_bad_id():
    pins.pin_align_rejects_bad_id()


@pytest.mark.parametrize("pin", pins.SHARD_PINS, ids=lambda f: f.__name__)
def test_shard_pin(pin):
    pin()


@pytest.mark.parametrize("pin", pins.SWIGLU_PINS, ids=lambda f: f.__name__)
def test_swiglu_pin(pin):
    pin()


@pytest.mark.parametrize("pin", pins.ROUTE_PINS, ids=lambda f: f.__name__)
def test_route_pin(pin):
    pin()
