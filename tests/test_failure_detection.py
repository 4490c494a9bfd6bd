"""Failure detection of the tcgen05 kernels, tested without faulting the GPU.

Every mbarrier wait in the kernels gives up after a time limit, records which wait gave up in a
status word (read and cleared by fa_device_status) and lets the kernel return, so the CUDA
context stays usable. The self-test entry point runs one such wait on a barrier that nothing
ever arrives on, with a short limit.
"""
import ctypes

import numpy as np
import pytest

from backward_adapter_gb300 import build as fbuild
from backward_adapter_gb300 import fa_train as ft
from backward_adapter_gb300 import workloads as wl


def test_selftest_rejects_out_of_range_limits():
    fbuild.build()
    lib = ft.load_library()
    assert lib.fa_train_selftest_wait(0, None) == ft.FA_ERR_INVALID_ARG
    assert lib.fa_train_selftest_wait(20000, None) == ft.FA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    import torch

    from tests import parity_util as pu

    ft.device_status()                       # start from a clear word
    ft.selftest_wait(50)
    torch.cuda.synchronize()                 # the kernel returned by itself
    assert ft.device_status() == (0x80000000 | ft.WAIT_SELFTEST_SITE)
    assert ft.device_status() == 0           # reading clears the word
    # the op still runs and still matches the oracle afterwards
    w = wl.Workload("after_selftest", B=1, Hq=2, Hkv=1, Sq=200, Sk=260, D=128, causal=True, q_offset=60, seed=51)
    inputs = wl.make_inputs(w)
    got = pu.run_gpu(w, pu.to_device(inputs, w))
    pu.assert_parity(w, got, pu.run_oracle(w, inputs))
