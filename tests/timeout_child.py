"""Child process of test_timeout_gpu.py (not collected by pytest: no test_ prefix).

Runs the bounded-wait timeout path of the kernels on the GPU with the test-only
library libfa_waittest.so, in which one launch may leave out one mbarrier
arrive (a barrier phase that nothing completes).  For each case: arm the
withheld arrive, make the call, read the raw device status word (wait site
<< 8 | status), then make the same call normally and compare it with the
fp64 oracle.  The parent sets FA_WAIT_TIMEOUT_MS (read once per process) so
that the waits run out quickly.  Prints one JSON line with the results.
"""
import ctypes
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from exact_io_aware_05_gb300 import build, inputs  # noqa: E402
from gpu_util import excess_over_output_rounding, to64  # noqa: E402

WITHHOLD_FWD_KV, WITHHOLD_FWD_EPI, WITHHOLD_BWD_DKV = 1, 2, 3


def main():
    lib = ctypes.CDLL(build.TEST_SO)
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp] * 5 + [i] * 6 + [fl, vp]
    lib.fa_bwd.argtypes = [vp] * 9 + [i] * 6 + [fl, vp, ctypes.c_size_t, vp]
    lib.fa_bwd_workspace_bytes.argtypes = [i] * 5
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_test_withhold.argtypes = [i]
    lib.fa_test_status_word.argtypes = [vp]
    lib.fa_sync_status.argtypes = [vp]
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda t: t.data_ptr()  # noqa: E731

    # one 256-row unit per CTA: B1 H1 T1024 d128 gives 4 forward units and 8 backward units,
    # each CTA 0 .. grid-1 takes one
    B, H, T, d = 1, 1, 1024, 128
    out = {}
    for name, which, causal in (("fwd_kv", WITHHOLD_FWD_KV, False), ("fwd_epi", WITHHOLD_FWD_EPI, True),
                                ("bwd_dkv", WITHHOLD_BWD_DKV, True)):
        w = inputs.small(B, H, T, T, d, causal, seed=41 + which, backward=True)
        x = inputs.generate(w, device="cuda")
        q, k, v, do = x["q"], x["k"], x["v"], x["do"]
        o = torch.empty_like(q)
        lse = torch.empty(B, H, T, device="cuda", dtype=torch.float32)

        def fwd():
            return lib.fa_fwd(p(q), p(k), p(v), p(o), p(lse), B, H, T, T, d, int(causal), w.scale, stream)

        res = {}
        if which != WITHHOLD_BWD_DKV:
            lib.fa_test_withhold(which)
            res["launch"] = fwd()
            res["word"] = lib.fa_test_status_word(stream)
            o.zero_()
            res["again_launch"] = fwd()
            res["again_status"] = lib.fa_sync_status(stream)
            o_ref, lse_ref = oracle.attention_fwd(to64(q[0, 0]), to64(k[0, 0]), to64(v[0, 0]), causal, w.scale)
            res["again_o_excess"] = excess_over_output_rounding(to64(o[0, 0]), o_ref)
            res["again_lse_err"] = float(np.abs(to64(lse[0, 0]) - lse_ref).max())
        else:
            assert fwd() == 0 and lib.fa_sync_status(stream) == 0
            ws = torch.empty(lib.fa_bwd_workspace_bytes(B, H, T, T, d), device="cuda", dtype=torch.uint8)
            dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))

            def bwd():
                return lib.fa_bwd(p(q), p(k), p(v), p(o), p(lse), p(do), p(dq), p(dk), p(dv), B, H, T, T, d,
                                  int(causal), w.scale, p(ws), ws.numel(), stream)

            lib.fa_test_withhold(which)
            res["launch"] = bwd()
            res["word"] = lib.fa_test_status_word(stream)
            for t in (dq, dk, dv):
                t.zero_()
            res["again_launch"] = bwd()
            res["again_status"] = lib.fa_sync_status(stream)
            g = oracle.attention_bwd(to64(q[0, 0]), to64(k[0, 0]), to64(v[0, 0]), to64(do[0, 0]), causal, w.scale)
            res["again_grad_excess"] = max(excess_over_output_rounding(to64(t[0, 0]), g[n])
                                           for n, t in (("dq", dq), ("dk", dk), ("dv", dv)))
        out[name] = res
    print(json.dumps(out))


if __name__ == "__main__":
    main()
