"""The failure path of the bounded device-side waits, taken without any GPU
fault: nvfp4_selftest_wait_timeout launches one thread that waits on an
mbarrier nothing completes.  The wait must give up after its cycle limit
(about 1.5 s), record NVFP4_ERR_TIMEOUT in the device status word and leave
the CUDA context usable.  Collected after the parity tests (it takes a
second or two) and before the no-alloc entry point's test, which comes
last."""
import time

import numpy as np
import pytest

import oracle
import synth
from nvfp4_testutil import to_dev, to_np_u8

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import nvfp4_weight_quantized_gb300 as nv  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_weight_quantized_gb300 import build
    build.build()
    nv.lib()


def test_bounded_wait_gives_up_and_reports_timeout():
    torch.cuda.synchronize()
    nv.nvfp4_get_device_status()  # clears whatever an earlier test left in the word
    t0 = time.perf_counter()
    nv.nvfp4_selftest_wait_timeout()
    assert nv.nvfp4_get_device_status() == nv.ERR_TIMEOUT  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert 0.2 < elapsed < 60, elapsed  # the wait ran to its limit, and ended
    assert nv.nvfp4_get_device_status() == nv.OK  # reading cleared it
    # the context is still usable: a quantisation right after matches the oracle
    w = synth.weight_normal(64, 256, seed=5)
    q = nv.nvfp4_quantize_fos(to_dev(w))
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == nv.OK
    assert np.array_equal(to_np_u8(q.codes), oracle.quantize_fos(w)["codes"])
