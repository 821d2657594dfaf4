"""Failure detection without a GPU fault: a kernel's bounded wait runs out on a
barrier nothing completes, the kernel records the timeout and returns, the
host reads SQ_ERR_DEVICE_TIMEOUT, and the context keeps working."""
import numpy as np
import pytest
import torch

import absmax_quantized_precision_gb300 as sq
import oracle
import synth
from gpu_util import DEV, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_stays_usable():
    torch.cuda.set_device(DEV)
    assert sq.sq_get_last_device_error() == sq.SQ_OK
    sq.sq_selftest_bounded_wait(20_000_000)            # 20 ms
    assert sq.sq_get_last_device_error() == sq.SQ_ERR_DEVICE_TIMEOUT
    assert sq.sq_get_last_device_error() == sq.SQ_OK   # read and cleared
    # the device still computes correctly afterwards
    x = synth.normal(91, (64, 256))
    q, s = sq.sq_quantize_rowwise_i8(to_dev(x))
    oq, osc = oracle.quantize_rowwise_i8(x)
    assert np.array_equal(q.cpu().numpy(), oq) and np.array_equal(s.cpu().numpy(), osc)
    assert sq.sq_get_last_device_error() == sq.SQ_OK


def test_selftest_rejects_unbounded_limits():
    with pytest.raises(sq.SQError):
        sq.sq_selftest_bounded_wait(0)
    with pytest.raises(sq.SQError):
        sq.sq_selftest_bounded_wait(10 ** 10)
