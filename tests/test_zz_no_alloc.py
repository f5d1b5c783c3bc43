"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (a plug-in whose host framework owns all device memory, or latency-
critical code that cannot take cudaMalloc's implicit synchronisation).  It
takes its scratch from a fixed array inside the library instead of a caller
workspace.  Called here through the C ABI (ctypes) and compared with fa_bwd on
the same inputs, twice in a row, because every call shares that array and must
not depend on what the previous call left in it.  Both run the same kernels, so
dk and dv must be bitwise equal and dq may differ only by the order in which
its fp32 reduce-adds landed.  The host-side checks (argument errors before the
scratch limit, sizes beyond it) need no GPU and live in test_abi.py.  This file
is collected last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import pytest
import torch

from exact_io_aware_05_gb300 import inputs
from gpu_util import assert_same_up_to_add_order

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.fa_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 9 + [i] * 6 + [ctypes.c_float, vp]
    f.restype = i
    return f


@pytest.mark.parametrize("B,H,T,d,causal", [(2, 4, 1000, 128, True), (1, 3, 700, 64, False)])
def test_noalloc_matches_fa_bwd_twice(B, H, T, d, causal):
    from exact_io_aware_05_gb300 import fa
    lib = ctypes.CDLL(fa.LIB_PATH)
    f = _noalloc(lib)
    w = inputs.small(B, H, T, T, d, causal, seed=31 + d, backward=True)
    x = inputs.generate(w, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o, lse = fa.attention_forward(q, k, v, causal, w.scale)
    ref = fa.attention_backward(q, k, v, o, lse, do, causal, w.scale)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
        st = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, T, T, d, int(causal), w.scale, stream)
        assert st == 0, fa.fa_status_string(st)
        assert fa.fa_sync_status() == fa.FA_OK
        assert torch.equal(dk, ref[1]), ("dk", call)
        assert torch.equal(dv, ref[2]), ("dv", call)
        assert_same_up_to_add_order(dq, ref[0], f"dq call {call}")
