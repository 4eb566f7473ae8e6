"""Both oracles against what the pages and mathematics fix (CPU only): the numpy
oracle and the C++ oracle answer the same pins through the same API."""
import pytest

from oracle import cpp_oracle
from oracle import q4_oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module", params=["numpy", "cpp"])
def oracle_impl(request):
    return q4_oracle if request.param == "numpy" else cpp_oracle.oracle()


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin, oracle_impl):
    pin(oracle_impl)
