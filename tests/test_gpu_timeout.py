"""The bounded-wait path of the f16/bf16 tensor-core kernel, made to run out
without faulting anything.

Every mbarrier wait in the tensor-core kernels gives up after a cycle limit:
the waiting thread sets the CTA's abort flag and the device status word, every
role drains what it started (copies in flight land, issued MMAs retire),
tensor memory is freed and the kernel returns.  The test hook
CONV2D_OVR_TEST_WITHHOLD makes CTA 0 skip the loads of its first pipeline
stage -- a barrier that nothing completes -- and CONV2D_OVR_TEST_WAIT_KCYCLES
shortens the limit to about 10 ms.  The call must come back, report
CONV2D_ERR_TIMEOUT through conv2d_get_device_status (read and cleared), and
the next normal call in the same process must be correct.
"""
import pytest
import torch

from cnn_convolution_gb300 import conv2d, workloads as wl
from parity import TOL, full_parity, run_gpu

pytestmark = pytest.mark.gpu

STATUS_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_convolution_gb300 import build
    import oracle
    build.build()
    conv2d.load()
    oracle.build()


@pytest.mark.parametrize("pair", [0, 1])
def test_withheld_stage_times_out_and_the_context_stays_usable(pair):
    # stride 2: the im2col kernel (the window kernel is for stride-1 layers);
    # pair=1: its 2-CTA variant, where CTA 0 is the pair's MMA issuer and the
    # odd CTA's copies of the withheld stage land on a barrier that never
    # completes
    spec = wl.ConvSpec("stall", 4, 64, 14, 14, 128, 3, 3, 2, 1, dtype="bf16", layout="NHWC")
    x, w, b = wl.random_inputs(spec, seed=3)
    assert conv2d.get_device_status() == 0
    with conv2d.overrides(test_withhold=1, test_wait_kcycles=20000, tc_cta2=pair):
        y, d = run_gpu(spec, x, w, b, "tensor_core")
        assert "a=im2col" in d.plan(), d.plan()
        assert (" cta2 " in d.plan()) == bool(pair), d.plan()
    assert conv2d.get_device_status() == STATUS_TIMEOUT
    assert conv2d.get_device_status() == 0          # read and cleared
    err = full_parity(spec, x, w, b, algo="tensor_core")
    assert err <= TOL["bf16"], err
    assert conv2d.get_device_status() == 0


@pytest.mark.parametrize("pair", [0, 1])
def test_short_wait_limit_alone_changes_nothing(pair):
    # the shortened limit without a withheld stage: every wait still succeeds
    spec = wl.ConvSpec("short_limit", 4, 64, 14, 14, 128, 3, 3, 2, 1, dtype="bf16", layout="NHWC")
    x, w, b = wl.random_inputs(spec, seed=4)
    with conv2d.overrides(test_wait_kcycles=20000, tc_cta2=pair):
        err = full_parity(spec, x, w, b, algo="tensor_core")
    assert err <= TOL["bf16"], err
    assert conv2d.get_device_status() == 0
