"""The allocation-free encode entry point against the handle-based one.

dflash_encode_noalloc serves callers that cannot call cudaMalloc (and so
cannot hand dflash_create a scratch area): its intermediates live in a static
device array.  Its output must match dflash_encode's on the same inputs,
within the encode tolerance the parity tests use (1e-4 of the largest |H_t|),
for two calls in a row (the second reuses the array the first one left
behind).  This file is collected last so that a failure here cannot hide any
other test's result; it also passes when run alone in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from block_diffusion_drafter_fc_gb300.synth import get_config, make_workload

pytestmark = pytest.mark.gpu


def test_encode_noalloc_matches_encode_twice():
    from block_diffusion_drafter_fc_gb300 import dflash as D
    fn = D.LIB.dflash_encode_noalloc
    fn.restype = C.c_int
    fn.argtypes = [C.POINTER(D.dflash_config), C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32,
                   C.c_void_p, C.c_void_p]
    wl = make_workload(get_config("small_bf16"))
    dw, feats = D.to_device(wl)
    dr = D.Drafter(wl.cfg, dw, max_inject=512)
    cfg = D.make_config(wl.cfg)
    stream = torch.cuda.current_stream().cuda_stream
    for (seq, p0, cnt, r0) in wl.inject_calls:          # 512 rows, then 37 rows
        f = feats[seq][r0:r0 + cnt]
        ref = torch.empty((cnt, wl.cfg.n_embd), dtype=torch.float32, device="cuda")
        dr.dflash_encode(f, ref)
        out = torch.full((cnt, wl.cfg.n_embd), float("nan"), dtype=torch.float32, device="cuda")
        rc = fn(C.byref(cfg), dw["fc"].data.data_ptr(), dw["hidden_norm"].data.data_ptr(),
                f.data_ptr(), cnt, out.data_ptr(), stream)
        assert rc == 0, D.LIB.dflash_status_string(rc).decode()
        torch.cuda.synchronize()
        a, b = out.cpu().numpy(), ref.cpu().numpy()
        assert np.isfinite(a).all()
        err = float(np.abs(a - b).max())
        assert err <= 1e-4 * float(np.abs(b).max()), err
    # a call beyond the static array's limit is rejected and launches nothing
    big = 16 * 16384 // ((wl.cfg.n_embd + 127) // 128) + 16
    assert fn(C.byref(cfg), dw["fc"].data.data_ptr(), dw["hidden_norm"].data.data_ptr(),
              feats[0].data_ptr(), big, out.data_ptr(), stream) == -3
    dr.close()
