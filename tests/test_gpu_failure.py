"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The tensor-core kernel bounds every barrier wait. Through the library's test
hook one hashing thread withholds its arrive at stage 0, so the MMA thread's
wait can never complete; with a 50 ms limit the kernel must record the timeout,
stop, free its tensor memory and return. The host reads VN_ERR_TIMEOUT from
vn_device_status(), the status clears, and the next ordinary call on the same
context is correct. Nothing here faults, traps or hangs the GPU."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import es
from tests.parity import TOL_BF16, assert_close, to_np
from virtual_noise_perturbed_gb300 import _lib, perturbed_linear_path, virtual_perturbed_linear
from virtual_noise_perturbed_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
P = ctypes.c_void_p


def test_bounded_wait_times_out_cleanly_and_context_stays_usable():
    build()
    lib = _lib.load()
    g = torch.Generator().manual_seed(3)
    pop, batch, in_f, out_f = 3, 32, 128, 128
    x = torch.randn(pop, batch, in_f, generator=g).to(torch.bfloat16).to(DEV)
    w = (torch.randn(out_f, in_f, generator=g) / in_f ** 0.5).to(torch.bfloat16).to(DEV)
    b = torch.zeros(out_f, dtype=torch.bfloat16, device=DEV)
    seeds = torch.arange(pop, dtype=torch.int64, device=DEV)
    y = torch.empty(pop, batch, out_f, dtype=torch.bfloat16, device=DEV)
    assert perturbed_linear_path(x, w) == "tc"
    stream = P(torch.cuda.current_stream().cuda_stream)
    assert lib.vn_device_status(stream) == _lib.VN_OK          # start clean

    st = lib.vn_testhook_linear_tc_withhold(
        P(x.data_ptr()), _lib.VN_BF16, 0, P(w.data_ptr()), _lib.VN_BF16, P(b.data_ptr()),
        _lib.VN_BF16, P(seeds.data_ptr()), pop, batch, in_f, out_f, 0.01, 0, P(y.data_ptr()),
        _lib.VN_BF16, 0, 50.0, stream)
    assert st == _lib.VN_OK                                    # launched
    assert lib.vn_device_status(stream) == 7                   # VN_ERR_TIMEOUT, read on the host
    assert lib.vn_device_status(stream) == _lib.VN_OK          # and cleared

    # The context is intact: an ordinary call right after is correct.
    y2 = virtual_perturbed_linear(x, w, b, seeds, 0.01, 0, path="tc")
    want = es.perturbed_linear(x.float().cpu().numpy(), w.float().cpu().numpy(),
                               b.float().cpu().numpy(), seeds.cpu().numpy(), 0.01, 0)
    assert_close(to_np(y2), want, TOL_BF16, "forward after a timed-out launch")
    assert lib.vn_device_status(stream) == _lib.VN_OK


def test_hook_refuses_bad_arguments():
    build()
    lib = _lib.load()
    z = P(0)
    assert lib.vn_testhook_linear_tc_withhold(z, 1, 0, z, 1, z, 1, z, 1, 32, 64, 64, 0.1, 0, z, 1,
                                               0, 0.0, z) == 4      # timeout must be > 0
    assert lib.vn_testhook_linear_tc_withhold(z, 1, 0, z, 1, z, 1, z, 1, 32, 64, 64, 0.1, 0, z, 1,
                                               -1, 10.0, z) == 4    # stage must be >= 0
