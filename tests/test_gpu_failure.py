"""Failure detection without a GPU fault: a device wait that nothing can satisfy gives up
after its bounded limit (about 2 s), the kernel reports GDN_DEVERR_TIMEOUT in the device
error word, the host reads it as GDN_ERR_TIMEOUT, and the context keeps working."""
import ctypes

import numpy as np
import pytest
import torch

from gated_deltanet_linear_conv1d_gb300 import synth
from tests import gdnutil as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gated_deltanet_linear_conv1d_gb300 import build
    build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding
    from tests.csrc import build_selftest
    st = ctypes.CDLL(build_selftest.build())
    st.bounded_wait_selftest.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    st.bounded_wait_selftest.restype = ctypes.c_int
    return binding, st


def test_a_wait_that_cannot_finish_times_out_and_the_context_survives(libs):
    b, st = libs
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert st.bounded_wait_selftest(err.data_ptr(), None) == 0
    host = ctypes.c_int32(0)
    status = b._lib.gdn_read_device_error(err.data_ptr(), ctypes.byref(host), 1, None)
    assert status == b.GDN_ERR_TIMEOUT
    assert host.value & b.GDN_DEVERR_TIMEOUT
    assert int(err.item()) == 0  # reset by the read
    # the context still runs real work: one decode step, checked against the oracle
    dims = synth.RANK_HEADS
    w = synth.decode_workload(dims, 4, 8, seed=71)
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    og = torch.zeros((4, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    b.gdn_decode_step(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"], d["alpha"], d["beta"],
                      d["z"], d["gamma"], w["eps"], ogate=og, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    r, _ = U.oracle_compact(w, np.arange(4))
    U.check_out(U.host_f64_from_bf16(og), r["ogate"], "ogate after the timeout")
