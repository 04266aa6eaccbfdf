"""The failure path of the bounded device waits, driven on purpose.

Every wait in the library has a time limit; when it runs out the kernel sets
a bit of the device status word and returns instead of waiting forever.  The
weight-resident chain (w4_chain_q4) waits on data other CTAs publish -- the
tagged outputs of the previous stage, and a grid barrier at each pass
boundary -- so its test entry point w4_chain_q4_test_timeout can make a wait
run out without any fault: one stage computes but never publishes its
outputs, and the limit is cut to a millisecond.  The stages that read those
outputs give up, and CTAs already waiting at the pass barrier give up on the
CTAs that left.  The test checks that the kernel returns, that the status
bit is set, and that the next normal call is clean and bit-exact.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from tests.test_gpu_microdecoder import _random_chain, oracle_chain
from w4a16_int4_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

STATUS_BARRIER_TIMEOUT = 4
K0 = 256
# depth 0: 256 rows; depth 1: 64 rows; depth 2: 64 rows; depth 3: 256 rows, the pass output.
# Small stages leave most CTAs without rows, so they go straight to the pass barrier.
SHAPES = [(256, -1), (64, 0), (64, 1), (256, 2)]


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_int4_quantized_gb300 import build
    build.build()
    from w4a16_int4_quantized_gb300 import ops as o
    o.device_status(clear=True)
    return o


def _check_clean_run(ops, ora, glins, olins, x0):
    ops.chain_q4(torch.from_numpy(x0).cuda(), glins, 2, 3)
    ref = oracle_chain(ora, x0, olins, 2, 3)
    torch.cuda.synchronize()
    for i, (_, _, y, _) in enumerate(glins):
        assert np.array_equal(y.cpu().numpy().view(np.uint32), ref[i].view(np.uint32)), i
    assert ops.device_status() == 0


@pytest.mark.parametrize("hold_stage", [1, 3, 5])
def test_held_stage_times_out_and_returns(ops, ora, hold_stage):
    """hold 1: a stage inside pass 0 (readers time out, CTAs at the pass
    barrier give up on them); hold 3: the pass output (pass 1 waits for it);
    hold 5: a stage of the last pass."""
    glins, olins = _random_chain(ops, ora, 4400, SHAPES, K0)
    x0 = synth.activations_f32(4401, 1, K0)
    ops.device_status(clear=True)
    t0 = time.perf_counter()
    st = ops.chain_q4_test_timeout(torch.from_numpy(x0).cuda(), glins, 2, 3, 1_000_000, hold_stage)
    assert st == ops.W4_OK
    torch.cuda.synchronize()  # the kernel returned
    elapsed = time.perf_counter() - t0
    assert elapsed < 0.5, elapsed  # a handful of 1 ms waits, not the 1 s default
    assert ops.device_status(clear=True) & STATUS_BARRIER_TIMEOUT
    # the held stage and those before it finished normally; a stage that gave
    # up left its output as the previous pass wrote it
    held_pass, held_depth = divmod(hold_stage, len(SHAPES))
    ref = [oracle_chain(ora, x0, olins, n, 3) for n in (1, 2)]
    for i in range(len(glins)):
        got = glins[i][2].cpu().numpy().view(np.uint32)
        if i <= held_depth:
            assert np.array_equal(got, ref[held_pass][i].view(np.uint32)), i
        elif held_pass >= 1:
            assert np.array_equal(got, ref[held_pass - 1][i].view(np.uint32)), i
    # the next normal call on the same device is clean and bit-exact
    _check_clean_run(ops, ora, glins, olins, x0)


def test_short_limit_without_hold_is_exact(ops, ora):
    glins, olins = _random_chain(ops, ora, 4410, SHAPES, K0)
    x0 = synth.activations_f32(4411, 1, K0)
    ops.device_status(clear=True)
    st = ops.chain_q4_test_timeout(torch.from_numpy(x0).cuda(), glins, 2, 3, 100_000_000, -1)
    assert st == ops.W4_OK
    ref = oracle_chain(ora, x0, olins, 2, 3)
    torch.cuda.synchronize()
    for i, (_, _, y, _) in enumerate(glins):
        assert np.array_equal(y.cpu().numpy().view(np.uint32), ref[i].view(np.uint32)), i
    assert ops.device_status() == 0


def test_timeout_arguments_checked_on_host(ops, ora):
    glins, _ = _random_chain(ops, ora, 4420, SHAPES, K0)
    x0 = torch.zeros(K0, device="cuda")
    assert ops.chain_q4_test_timeout(x0, glins, 1, 3, 0, -1) == ops.W4_EINVAL
    assert ops.chain_q4_test_timeout(x0, glins, 1, 3, 2_000_000_000, -1) == ops.W4_EINVAL
    assert ops.chain_q4_test_timeout(x0, glins, 1, 3, 1_000_000, -2) == ops.W4_EINVAL
    torch.cuda.synchronize()
    assert ops.device_status() == 0
