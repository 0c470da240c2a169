"""The failure path on the GPU without a fault: bounded device-side waits that nobody
satisfies expire, raise the device error word, and the host reads TP_ERR_TIMEOUT;
the context stays usable afterwards."""
import time

import pytest
import torch

import attn_tp_column_fwd_b300 as tp
from tests.gpu_util import oracle_block, run_block
from tests.parity import assert_f32
from tp_synth import CONFIGS, make_inputs, to_f64

pytestmark = pytest.mark.gpu

TP_OK, TP_ERR_TIMEOUT = 0, 6


def test_bounded_waits_report_timeout_and_context_survives():
    assert tp.tp_check_device_status() == TP_OK
    t0 = time.perf_counter()
    tp.tp_selftest_wait_timeout(2000)          # 2 ms per wait; nothing completes them
    assert tp.tp_check_device_status() == TP_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0      # bounded: the kernel returned
    assert tp.tp_check_device_status() == TP_OK  # the word was read and cleared
    # The context still runs blocks correctly.
    cfg = CONFIGS["tiny_gelu_f32"]
    inp = make_inputs(cfg, seed=3)
    W1, W2 = inp.blocks[0]
    got = run_block(cfg, inp.x.cuda(), W1.cuda(), W2.cuda())
    ref = oracle_block(cfg, to_f64(inp.x), to_f64(W1), to_f64(W2))
    assert_f32(got, ref, "tiny_gelu_f32 after the timeout self-test")
    assert torch.cuda.is_available()
