"""The synthetic weight quantizers (harness steps, not part of the drafter): the
FP4 buffer layout and round-trip error, decoded by the oracle."""
import numpy as np
import torch

from block_diffusion_drafter_fc_gb300 import synth as S
from oracle import dflash_oracle as O


def test_fp4_buffer_size_and_roundtrip_error():
    g = torch.Generator().manual_seed(0)
    w = torch.randn(37, 512, generator=g) * 0.02
    q, s = S.quantize_fp4_rows(w)
    assert q.dtype == torch.uint8 and q.numel() == S.fp4_nbytes(37, 512) == 37 * 256 + 48 * 32
    d = O.decode(q.numpy(), "fp4", s.numpy())
    wb = w.double().numpy().reshape(37, 32, 16)
    amax = np.abs(wb).max(axis=2)
    # E2M1 steps are at most 2 between 4 and 6 (half a step = 1/6 of the block
    # maximum) plus the E4M3 rounding of the block scale (2^-4 relative)
    err = np.abs(d.reshape(37, 32, 16) - wb).max(axis=2) / amax
    assert err.max() <= 1 / 6 * (1 + 2 ** -4) + 2 ** -4


def test_fp4_exact_grid_roundtrips():
    """Weights that are already E2M1 values times a power-of-two block scale (the
    block maximum 6 x scale) come back up to the f32 rounding of the row scale."""
    g = np.random.default_rng(1)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    n, k = 20, 256
    v = grid[g.integers(0, 8, size=(n, k))] * np.where(g.random((n, k)) < 0.5, -1, 1)
    v.reshape(n, k // 16, 16)[:, :, 0] = 6.0          # every block reaches 6
    bscale = 2.0 ** g.integers(-3, 3, size=(n, k // 16))
    w = v * np.repeat(bscale, 16, axis=1) * 2.0 ** -7
    q, s = S.quantize_fp4_rows(torch.from_numpy(w).float())
    d = O.decode(q.numpy(), "fp4", s.numpy())
    assert np.all(np.abs(d - w) <= 2.0 ** -22 * np.abs(w))
    assert np.array_equal(d == 0, w == 0)


def test_fp4_zero_rows():
    w = torch.zeros(3, 64)
    w[1, 5] = 0.25
    q, s = S.quantize_fp4_rows(w)
    d = O.decode(q.numpy(), "fp4", s.numpy())
    assert s[0] == 1.0 and s[2] == 1.0
    assert np.array_equal(d[[0, 2]], np.zeros((2, 64)))
    assert abs(d[1, 5] - 0.25) <= 2.0 ** -22 and np.count_nonzero(d[1]) == 1


def test_fp8_rows_scale_and_error():
    """E4M3 row quantizer: s = max|w_row| / 448 (1 for an all-zero row), the row
    maximum maps to code +-448 exactly, and every weight is within half an E4M3
    step (2^-4 relative for normal values, 2^-10 s absolute below them)."""
    g = torch.Generator().manual_seed(3)
    w = torch.randn(9, 300, generator=g) * 0.05
    w[4] = 0.0
    q, s = S.quantize_fp8_rows(w)
    assert q.dtype == torch.uint8 and s.dtype == torch.float32
    amax = w.abs().amax(dim=1)
    assert s[4] == 1.0
    for r in (0, 1, 2, 3, 5, 6, 7, 8):
        assert s[r] == (amax[r] / 448).float()
    d = O.decode(q.numpy(), "fp8", s.numpy())
    wd = w.double().numpy()
    sc = s.double().numpy()[:, None]
    assert np.all(np.abs(d) <= 448 * sc + 1e-30)
    rel_ok = np.abs(d - wd) <= 2.0 ** -4 * np.abs(wd) + 2.0 ** -10 * sc
    assert rel_ok.all()
    assert np.all(d[4] == 0)


def test_workload_is_deterministic_and_follows_the_schedule():
    cfg = S.get_config("tiny_f32")
    a, b = S.make_workload(cfg), S.make_workload(cfg)
    for name in a.weights:
        assert torch.equal(a.weights[name].data, b.weights[name].data), name
    assert all(torch.equal(x, y) for x, y in zip(a.feats, b.feats))
    assert torch.equal(a.id_last, b.id_last) and torch.equal(a.mismatch, b.mismatch)
    # inject positions 0..63, then 64..79 (wrapping the 64-slot window); block at 80
    assert a.inject_calls == [(0, 0, 64, 0), (0, 64, 16, 64)]
    assert a.n_past.tolist() == [80]
    assert a.feats[0].shape == (80, cfg.feat_dim) and a.feats[0].dtype == torch.float32
    assert 0 <= int(a.id_last[0]) < cfg.n_vocab and 0 <= int(a.mismatch[0]) <= 15
    small = S.get_config("small_bf16")
    assert small.inject == ((0, 512), (512, 37)) and small.window == 512
    real = S.get_config("real_bf16")
    assert real.inject == ((0, 2048),) and real.window == 2048


def test_batched_fills_offsets_and_positions():
    cfg = S.get_config("ragged_bf16")
    wl = S.make_workload(cfg)
    assert len(wl.fills) == len(wl.offsets) == cfg.n_seq
    for s in range(cfg.n_seq):
        f, o = wl.fills[s], wl.offsets[s]
        assert cfg.fill_lo <= f <= cfg.fill_hi and 0 <= o <= cfg.offset_hi
        assert wl.inject_calls[s] == (s, o, f, 0)
        assert int(wl.n_past[s]) == o + f
        assert wl.positions(wl.inject_calls[s]).tolist() == list(range(o, o + f))
        assert wl.feats[s].shape == (f, cfg.feat_dim)


def test_targets_put_the_first_mismatch_at_the_drawn_index():
    """make_targets: accept() of the drafts against the targets returns exactly
    the drawn mismatch index (15 = the whole block agrees), whatever the tail."""
    g = np.random.default_rng(5)
    V = 50
    drafts = g.integers(0, V, size=(64, 15)).astype(np.int32)
    m = np.concatenate([np.arange(16), g.integers(0, 16, size=48)]).astype(np.int32)
    tail = g.integers(0, V, size=(64, 15)).astype(np.int32)
    t = S.make_targets(drafts, m, tail, V)
    assert t.dtype == np.int32 and t.shape == (64, 15)
    assert np.array_equal(O.accept(drafts, t), m)
    for s in range(64):
        if m[s] < 15:
            assert t[s, m[s]] == (drafts[s, m[s]] + 1) % V
            assert np.array_equal(t[s, m[s] + 1:], tail[s, m[s] + 1:])
