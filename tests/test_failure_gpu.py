"""The failure path of the kernels' bounded waits, exercised on the GPU
without a fault: a kernel whose wait nothing completes gives up after its
limit, records FD_ERR_DEVICE_TIMEOUT in the device status word, and ends;
the context stays usable and the next decode is correct."""
import time

import numpy as np
import pytest
import torch

import oracle
import split_kv_fd_gb300 as fd
from split_kv_fd_gb300.inputs import random_case
from parity_util import check_lse, check_out

pytestmark = pytest.mark.gpu

FD_ERR_DEVICE_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    fd.load()
    fd.device_status(reset=True)
    yield
    assert fd.device_status() == 0


def test_bounded_wait_gives_up_and_reports():
    assert fd.device_status(reset=True) == 0
    t0 = time.perf_counter()
    fd.selftest_wait_timeout()                 # the kernels' limit: 1 s
    got = fd.device_status(reset=True)         # synchronises
    waited = time.perf_counter() - t0
    assert got == FD_ERR_DEVICE_TIMEOUT
    assert waited >= 0.9                       # it did wait for its limit
    assert waited < 10.0                       # and then gave up
    assert fd.device_status() == 0             # the reset cleared it


def test_context_usable_after_a_timeout():
    fd.selftest_wait_timeout()
    assert fd.device_status(reset=True) == FD_ERR_DEVICE_TIMEOUT
    q, k, v, lens = random_case(2, 4, 600, 128, "bf16", lens=[600, 217], seed=31)
    ref_out, ref_lse = oracle.attention(q, k, v, lens=lens)
    dev = torch.device("cuda")
    out, lse = fd.decode(q.to(dev), k.to(dev), v.to(dev), lens.to(dev), out_dtype=torch.float32)
    check_out(out, ref_out, "bf16")
    check_lse(lse, ref_lse, "bf16")
    assert fd.device_status() == 0

