"""Failure detection without a GPU fault (needs a GB300).

The kernels bound every pipeline wait. A testing hook makes the next launches
leave one pipeline stage unfilled, so the MMA issuer's wait on it runs out
after a short limit; the kernel then stops cleanly (in-flight copies and MMAs
drained, tensor memory released) and the host reads SWIGLU_ERR_TIMEOUT from
the status word. The context must stay usable: the next normal call is
checked against the oracle.
"""
import pytest
import torch

from gpu_helpers import check_against_oracle, to_dev
from swiglu_gated_mlp_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native(native_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return native_lib


@pytest.mark.parametrize("variant,M", [(1, 64), (2, 16), (1, 300), (3, 300), (4, 200), (5, 128)])
def test_stalled_pipeline_reports_timeout_and_context_survives(native, variant, M):
    K, N = 256, 384
    a, w1, w2 = make_inputs(M, K, N, seed=5)
    ad, w1d, w2d = to_dev(a, w1, w2)
    wp = native.swiglu_pack_weights(w1d, w2d)
    native.swiglu_check_device_status()
    native.swiglu_testing_inject_stall(True, timeout_ms=200)
    try:
        native.swiglu_forward_variant(ad, wp, N, variant)
        with pytest.raises(native.SwigluError) as err:
            native.swiglu_check_device_status()
        assert err.value.code == native.SWIGLU_ERR_TIMEOUT
    finally:
        native.swiglu_testing_inject_stall(False, timeout_ms=1000)
    native.swiglu_check_device_status()  # cleared by the previous read
    check_against_oracle(native, M, K, N, seed=5, variant=variant)
