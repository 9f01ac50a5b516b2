"""The oracle against facts fixed by the mathematics (CPU only)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_thread_count_does_not_change_result(oracle_lib):
    import numpy as np
    import oracle
    r, w, k, v, kk, a = oracle_pins._draw(13, 5, 8, seed=99)
    cu = np.array([0, 4, 13])
    o1, s1 = oracle.run(r, w, k, v, kk, a, cu_seqlens=cu, nthreads=1, lib=oracle_lib)
    o2, s2 = oracle.run(r, w, k, v, kk, a, cu_seqlens=cu, nthreads=7, lib=oracle_lib)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_rejects_malformed_cu_seqlens(oracle_lib):
    import numpy as np
    import oracle
    r, w, k, v, kk, a = oracle_pins._draw(5, 1, 4, seed=98)
    with pytest.raises(ValueError):
        oracle.run(r, w, k, v, kk, a, cu_seqlens=np.array([0, 4, 3, 5]), lib=oracle_lib)
