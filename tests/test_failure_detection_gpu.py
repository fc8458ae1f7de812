"""Failure detection on the GPU without a fault: a wait that nothing satisfies gives up
after its time limit, the device status word reports FA_ERR_DEVICE_TIMEOUT, the word is
cleared by reading it, and the context keeps working."""
import math

import pytest
import torch

from exact_attention_tmem_gb300 import _lib, inputs
from gpu_helpers import assert_fwd_close, gpu_fwd, oracle_fwd

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_is_reported():
    import exact_attention_tmem_gb300 as fa
    fa.build()
    lib = _lib.load()
    stream = torch.cuda.current_stream()
    assert fa.device_status() == _lib.FA_OK
    assert lib.fa_selftest_wait_timeout(stream.cuda_stream) == _lib.FA_OK
    assert lib.fa_get_device_status(stream.cuda_stream) == _lib.FA_ERR_DEVICE_TIMEOUT
    assert lib.fa_get_device_status(stream.cuda_stream) == _lib.FA_OK      # read clears it
    # the context is still usable: a normal call afterwards is correct
    q, k, v = inputs.random_inputs(1, 2, 300, 128, seed=99)
    o, lse = gpu_fwd(q, k, v, True)
    o_ref, l_ref = oracle_fwd(q, k, v, True, 1.0 / math.sqrt(128))
    assert_fwd_close(o, lse, o_ref, l_ref, "after a reported timeout")
