"""The read-rate measurement aid (moe_measure_read_rate) through the C ABI:
it runs, returns a rate between zero and well above any HBM peak, and
rejects bad arguments."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


def test_read_rate_runs_and_is_plausible():
    from expert_cache_serving_gb300 import moecache as mc

    nbytes, n_bufs = 64 << 20, 4
    buf = torch.ones(n_bufs * nbytes, dtype=torch.uint8, device="cuda")
    g = mc.moe_measure_read_rate(buf, nbytes, n_bufs, 8, torch.cuda.current_stream())
    assert 100.0 < g < 20000.0


def test_read_rate_rejects_bad_arguments():
    import ctypes

    from expert_cache_serving_gb300 import moecache as mc

    buf = torch.ones(1 << 20, dtype=torch.uint8, device="cuda")
    g = ctypes.c_double()
    assert mc.lib.moe_measure_read_rate(buf.data_ptr(), 1000, 1, 1, None, ctypes.byref(g)) == mc.MOE_ERR_INVALID_ARG
    assert mc.lib.moe_measure_read_rate(buf.data_ptr() + 8, 1024, 1, 1, None, ctypes.byref(g)) == mc.MOE_ERR_INVALID_ARG
    assert mc.lib.moe_measure_read_rate(buf.data_ptr(), 1024, 0, 1, None, ctypes.byref(g)) == mc.MOE_ERR_INVALID_ARG
    assert mc.lib.moe_measure_read_rate(None, 1024, 1, 1, None, ctypes.byref(g)) == mc.MOE_ERR_INVALID_ARG
