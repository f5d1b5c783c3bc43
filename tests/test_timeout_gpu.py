"""The device-side timeout path, run on the GPU without a fault.

Every spin-wait in the kernels is bounded: when one runs out, its role raises
the CTA's abort flag and records (wait site << 8 | FA_ERR_TIMEOUT) in the
kernel's status word; every role then leaves its loop, waits for the copies
and MMAs it has in flight, tensor memory is freed and the kernel returns.
Here a test-only build of the library (libfa_waittest.so, compiled with
FA_TEST_WITHHOLD=1; libfa.so has none of it) leaves out one mbarrier arrive in
one launch, so that a barrier phase is never completed, with a 250 ms limit.
The test checks that the call returns, that the status word names a wait the
withheld arrive blocks, that the status is then clear, and that the same call
made normally right after matches the oracle.  Run in a child process, because
the wait limit is read once per process.
"""
import json
import os
import subprocess
import sys

import pytest

from gpu_util import TOL_GRAD, TOL_LSE, TOL_O_BF16

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
FA_ERR_TIMEOUT = 4
# wait sites (the second byte of the status word), as numbered in the kernels
FWD_P_EMPTY, FWD_M_FULL, FWD_S_SFULL, FWD_S_EPI = 1, 4, 7, 9
BWD_D_DKVFULL = 12


@pytest.fixture(scope="module")
def results():
    from exact_io_aware_05_gb300 import build
    build.build(test_variant=True)
    env = dict(os.environ, FA_WAIT_TIMEOUT_MS="250")
    r = subprocess.run([sys.executable, os.path.join(HERE, "timeout_child.py")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def _check(res, sites):
    assert res["launch"] == 0
    word = res["word"]
    assert word & 0xFF == FA_ERR_TIMEOUT, hex(word)
    assert (word >> 8) in sites, hex(word)
    assert res["again_launch"] == 0 and res["again_status"] == 0


def test_forward_kv_slot_never_released(results):
    """Tile 0 of CTA 0 keeps its first K/V slot: the producer's wait for that slot runs out,
    or first the MMA issuers' or the softmax's waits for the copies the producer cannot
    make; which one reaches its limit first depends on the polling."""
    res = results["fwd_kv"]
    _check(res, {FWD_P_EMPTY, FWD_M_FULL, FWD_S_SFULL})
    assert res["again_o_excess"] <= TOL_O_BF16 and res["again_lse_err"] <= TOL_LSE


def test_forward_epilogue_never_signalled(results):
    """Tile 0 of CTA 0 never gets its final O~: only its softmax waits for it."""
    res = results["fwd_epi"]
    _check(res, {FWD_S_EPI})
    assert res["again_o_excess"] <= TOL_O_BF16 and res["again_lse_err"] <= TOL_LSE


def test_backward_dkv_never_signalled(results):
    """CTA 0's dK, dV are never signalled complete: only the drain warpgroup waits for them."""
    res = results["bwd_dkv"]
    _check(res, {BWD_D_DKVFULL})
    assert res["again_grad_excess"] <= TOL_GRAD
