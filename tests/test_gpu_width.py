"""Narrow blocks (dflash_set_block_width; dflash_head.rs, set_block_g: the
anchor plus num_drafts mask rows, 2..16 rows, one captured graph per width)
against the oracle's step over a block of the same width.

Logits of the B existing rows within the storage tolerance, drafts 0..B-2
equal outside near ties and -1 beyond, acceptance counts bit-exact (at most
B-1), and per-width graphs that replay bitwise like the eager step."""
import numpy as np
import pytest
import torch

from block_diffusion_drafter_fc_gb300.synth import BLOCK, get_config, make_targets, make_workload
import gpu_harness as GH
import oracle_bridge as OB
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_f32", "ragged_bf16", "small_fp8", "small_fp4"])
def test_block_width_matches_oracle(name):
    from block_diffusion_drafter_fc_gb300 import dflash as D
    cfg = get_config(name)
    wl = make_workload(cfg)
    n = cfg.n_seq
    w, rings, _ = OB.oracle_prefill(wl)
    idl, npast = wl.id_last.numpy()[:n], wl.n_past.numpy()[:n]
    dw, feats = GH.to_device(wl, "cuda")
    dr = D.Drafter(cfg, dw, max_seq=n, max_inject=max(c[2] for c in wl.inject_calls))
    GH.prefill(dr, wl, feats)
    id_last, n_past = wl.id_last[:n].cuda(), wl.n_past[:n].cuda()
    logits = torch.empty((n, BLOCK, cfg.n_vocab), device="cuda")
    drafts = torch.empty((n, BLOCK - 1), dtype=torch.int32, device="cuda")
    n_ok = torch.empty((n,), dtype=torch.int32, device="cuda")
    tol = GH.logit_tol(cfg)
    g = torch.Generator().manual_seed(4242 + cfg.seed)
    eager = {}
    for B in (2, 5, 16):
        ref_logits, ref_drafts = O.step(w, rings, idl, npast, width=B)
        dr.dflash_set_block_width(B)
        dr.dflash_step(id_last, n_past, logits, drafts)
        torch.cuda.synchronize()
        lg, dd = logits.cpu().numpy(), drafts.cpu().numpy()
        err = float(np.max(np.abs(lg[:, :B] - ref_logits)))
        assert err <= tol, f"width {B}: logits max |diff| {err:.3e}"
        GH.compare_drafts(lg[:, :B], dd[:, :B - 1], ref_logits, ref_drafts, err, name)
        assert (dd[:, B - 1:] == -1).all(), f"width {B}: drafts past the block"
        # acceptance: the target agrees with the oracle's drafts up to a drawn m <= B-1
        m = torch.randint(0, B, (n,), generator=g).numpy()
        tail = torch.randint(0, cfg.n_vocab, (n, BLOCK - 1), generator=g).numpy()
        padded = np.full((n, BLOCK - 1), -1, dtype=np.int64)
        padded[:, :B - 1] = ref_drafts
        targets = make_targets(np.where(padded < 0, 0, padded), np.minimum(m, BLOCK - 1), tail,
                               cfg.n_vocab)
        want = O.accept(ref_drafts, targets[:, :B - 1])
        dr.dflash_accept(drafts, torch.from_numpy(targets).cuda(), n_ok)
        if not GH.compare_drafts(lg[:, :B], dd[:, :B - 1], ref_logits, ref_drafts, err, name):
            assert np.array_equal(n_ok.cpu().numpy(), want), f"width {B}: n_ok"
        eager[B] = (lg.copy(), dd.copy())
    # one graph per width, replayed alternately: bitwise equal to the eager steps
    for B in (5, 16):
        dr.dflash_set_block_width(B)
        dr.dflash_capture(id_last, n_past, logits, drafts)
    for B in (5, 16, 5):
        dr.dflash_set_block_width(B)
        dr.dflash_replay()
        torch.cuda.synchronize()
        assert np.array_equal(logits.cpu().numpy()[:, :B], eager[B][0][:, :B]), B
        assert np.array_equal(drafts.cpu().numpy(), eager[B][1]), B
    assert dr.dflash_read_status() == 0
    with pytest.raises(D.DFlashError):
        dr.dflash_set_block_width(1)
    with pytest.raises(D.DFlashError):
        dr.dflash_set_block_width(17)
    dr.close()
