"""The allocation-free encode entry point (dflash_encode_noalloc).

Some callers cannot call cudaMalloc: code inside an allocator-free runtime, a
plug-in that may only touch the buffers it is handed, a host whose device
memory all belongs to a pool.  They cannot give dflash_create its scratch
area, so this encode keeps its intermediates in a static device array.

Checked here, each on two calls in a row (the second reuses the array the
first left behind):
  * against the fp64 oracle's encode and against the handle-based
    dflash_encode on the same inputs, within the encode tolerance of the parity
    tests (1e-4 of the largest |H_t|), for fp32 features and weights
    (tiny_f32) and for bf16 (small_bf16);
  * at the largest accepted row count for the real drafter width (n_embd
    6656: T = 5040), sampled rows against the oracle;
  * one row past the limit returns DFLASH_ERR_TOO_MANY_ROWS, with buffers that
    really hold that many rows, so even a wrong answer touches no memory
    outside them.
This file is collected last so that a failure here cannot hide any other
test's result; it also passes when run alone in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from block_diffusion_drafter_fc_gb300.synth import get_config, make_workload, raw_numpy
import gpu_harness as GH
import oracle_bridge as OB

pytestmark = pytest.mark.gpu

TOO_MANY_ROWS = -3


def _noalloc(cfg_c, fc, hidden_norm, feats, T, out):
    from block_diffusion_drafter_fc_gb300 import dflash as D
    stream = torch.cuda.current_stream().cuda_stream
    return D.LIB.dflash_encode_noalloc(C.byref(cfg_c), fc.data_ptr(), hidden_norm.data_ptr(),
                                       feats.data_ptr(), T, out.data_ptr(), stream)


def _close(a, b):
    err = float(np.abs(a - b).max())
    assert err <= 1e-4 * float(np.abs(b).max()), err


@pytest.mark.parametrize("name", ["tiny_f32", "small_bf16"])
def test_encode_noalloc_matches_oracle_and_encode(name):
    from block_diffusion_drafter_fc_gb300 import dflash as D
    from oracle import dflash_oracle as O
    wl = make_workload(get_config(name))
    w = OB.oracle_weights(wl)
    dw, feats = GH.to_device(wl)
    dr = D.Drafter(wl.cfg, dw, max_inject=max(c[2] for c in wl.inject_calls))
    cfg_c = D.make_config(wl.cfg)
    for call in wl.inject_calls:          # e.g. 512 rows, then 37 rows
        seq, _, cnt, r0 = call
        f = feats[seq][r0:r0 + cnt]
        ref = torch.empty((cnt, wl.cfg.n_embd), dtype=torch.float32, device="cuda")
        dr.dflash_encode(f, ref)
        out = torch.full((cnt, wl.cfg.n_embd), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(cfg_c, dw["fc"].data, dw["hidden_norm"].data, f, cnt, out)
        assert rc == 0, D.LIB.dflash_status_string(rc).decode()
        torch.cuda.synchronize()
        a = out.cpu().numpy()
        assert np.isfinite(a).all()
        _close(a, O.encode(w, raw_numpy(wl.call_feats(call))))
        _close(a, ref.cpu().numpy())
    dr.close()


def test_encode_noalloc_limits_at_real_width():
    from block_diffusion_drafter_fc_gb300 import dflash as D
    from oracle import dflash_oracle as O
    cfg = get_config("real_bf16")
    d, fdim = cfg.n_embd, cfg.feat_dim
    tiles = (d + 127) // 128
    t_max = 16384 // tiles * 16                      # 5040 rows at n_embd 6656
    g = torch.Generator().manual_seed(77)
    fc = (torch.randn(d, fdim, generator=g) / fdim ** 0.5).to(torch.bfloat16)
    hn = (1 + 0.02 * torch.randn(d, generator=g)).to(torch.bfloat16)
    feats = torch.randn(t_max + 1, fdim, generator=g).to(torch.bfloat16)
    fc_d, hn_d, feats_d = fc.cuda(), hn.cuda(), feats.cuda()
    out = torch.zeros((t_max + 1, d), dtype=torch.float32, device="cuda")
    cfg_c = D.make_config(cfg)
    w = O.OracleWeights(OB.oracle_config(cfg), {"fc": raw_numpy(fc), "hidden_norm": raw_numpy(hn)})
    rows = np.array([0, 1, 17, 2047, 4000, t_max - 1])
    want = O.encode(w, raw_numpy(feats[torch.from_numpy(rows)]))
    for _ in range(2):
        out.fill_(float("nan"))
        assert _noalloc(cfg_c, fc_d, hn_d, feats_d, t_max, out) == 0
        torch.cuda.synchronize()
        a = out[:t_max].cpu().numpy()
        assert np.isfinite(a).all()
        _close(a[rows], want)
    # one row more is beyond the static array's limit: rejected, nothing launched
    out.fill_(-7.0)
    assert _noalloc(cfg_c, fc_d, hn_d, feats_d, t_max + 1, out) == TOO_MANY_ROWS
    torch.cuda.synchronize()
    assert bool((out == -7.0).all())


def test_encode_noalloc_rejects_past_limit_small_width():
    """n_embd 2048 (16 tiles): 16384 rows are accepted by the ticket limit, 16385
    are not; the buffers hold 16385 rows."""
    from block_diffusion_drafter_fc_gb300 import dflash as D
    cfg = get_config("small_bf16")
    big = 16 * 16384 // ((cfg.n_embd + 127) // 128) + 1
    feats = torch.zeros((big, cfg.feat_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((big, cfg.n_embd), dtype=torch.float32, device="cuda")
    fc = torch.zeros((cfg.n_embd, cfg.feat_dim), dtype=torch.bfloat16, device="cuda")
    hn = torch.ones((cfg.n_embd,), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(D.make_config(cfg), fc, hn, feats, big, out) == TOO_MANY_ROWS
