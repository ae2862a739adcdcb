"""The device-resident speculative loop (dflash_advance, dflash_capture_loop)
against the oracle's loop turn (oracle.advance + oracle.step) on the same
seeded inputs.

Each turn: the target's tokens for the 16 block rows are built from the
oracle's drafts with a drawn first mismatch (uniform in 0..15; 15 = all
accepted) and its features are seeded random values in the storage dtype.
Both sides advance from the same drafts (the oracle's, copied into the
device buffer), so acceptance counts, next anchors, positions and ring slot
positions must be bit-exact; logits within the storage tolerance; drafts
equal outside near ties.  Two eager turns, then two turns replayed from the
captured loop graph.
"""
import numpy as np
import pytest
import torch

from block_diffusion_drafter_fc_gb300.synth import BLOCK, get_config, make_targets, make_workload, raw_numpy
import gpu_harness as GH
import oracle_bridge as OB
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _turn_inputs(cfg, ref_drafts, turn):
    g = torch.Generator().manual_seed(7000 + 31 * turn + cfg.seed)
    n = ref_drafts.shape[0]
    mism = torch.randint(0, BLOCK, (n,), generator=g).numpy()
    tail = torch.randint(0, cfg.n_vocab, (n, BLOCK - 1), generator=g).numpy()
    t15 = make_targets(ref_drafts, mism, tail, cfg.n_vocab)
    bonus = torch.randint(0, cfg.n_vocab, (n, 1), generator=g).numpy().astype(np.int32)
    targets = np.concatenate([t15, bonus], axis=1).astype(np.int32)
    feats = torch.randn((n, BLOCK, cfg.feat_dim), generator=g).to(TORCH_DT[cfg.dense_dtype])
    return targets, feats


@pytest.mark.parametrize("name", ["tiny_f32", "ragged_bf16", "small_fp8", "many_seq_bf16", "small_fp4"])
def test_loop_turns_match_oracle(name):
    from block_diffusion_drafter_fc_gb300 import dflash as D
    cfg = get_config(name)
    wl = make_workload(cfg)
    n = cfg.n_seq
    w, rings, _ = OB.oracle_prefill(wl)
    idl, npast = wl.id_last.numpy()[:n].astype(np.int32), wl.n_past.numpy()[:n].astype(np.int32)
    ref_logits, ref_drafts = O.step(w, rings, idl, npast)

    dw, feats0 = GH.to_device(wl, "cuda")
    max_inject = max(max(c[2] for c in wl.inject_calls), BLOCK * n)
    dr = D.Drafter(cfg, dw, max_seq=n, max_inject=max_inject)
    GH.prefill(dr, wl, feats0)
    id_last = wl.id_last[:n].cuda()
    n_past = wl.n_past[:n].cuda()
    logits = torch.empty((n, BLOCK, cfg.n_vocab), device="cuda")
    drafts = torch.empty((n, BLOCK - 1), dtype=torch.int32, device="cuda")
    n_ok = torch.empty((n,), dtype=torch.int32, device="cuda")
    targets_d = torch.empty((n, BLOCK), dtype=torch.int32, device="cuda")
    feats_d = torch.empty((n, BLOCK, cfg.feat_dim), dtype=TORCH_DT[cfg.dense_dtype], device="cuda")
    dr.dflash_step(id_last, n_past, logits, drafts)
    tol = GH.logit_tol(cfg)

    def check(turn, ref_nok):
        torch.cuda.synchronize()
        lg = logits.cpu().numpy()
        err = float(np.max(np.abs(lg - ref_logits)))
        assert err <= tol, f"turn {turn}: logits max |diff| {err:.3e} > {tol}"
        GH.compare_drafts(lg, drafts.cpu().numpy(), ref_logits, ref_drafts, err, name)
        if ref_nok is not None:
            assert np.array_equal(n_ok.cpu().numpy(), ref_nok), turn
        assert np.array_equal(id_last.cpu().numpy(), idl), turn
        assert np.array_equal(n_past.cpu().numpy(), npast), turn
        _, _, pos = dr.ring_views()
        for s in range(n):
            assert np.array_equal(pos[s].cpu().numpy(), rings[s].pos), (turn, s)
        assert dr.dflash_read_status() == 0

    check(-1, None)
    prev_drafts = ref_drafts
    for turn in range(4):
        targets, feats = _turn_inputs(cfg, prev_drafts, turn)
        ref_nok, idl, npast = O.advance(w, rings, prev_drafts, targets, raw_numpy(feats), idl, npast)
        ref_logits, ref_drafts = O.step(w, rings, idl, npast)
        # both sides advance from the same drafts: the oracle's of the previous step
        drafts.copy_(torch.from_numpy(np.ascontiguousarray(prev_drafts)))
        targets_d.copy_(torch.from_numpy(targets))
        feats_d.copy_(feats)
        if turn < 2:
            dr.dflash_advance(drafts, targets_d, feats_d, id_last, n_past, n_ok)
            dr.dflash_step(id_last, n_past, logits, drafts)
        else:
            if turn == 2:
                # a plain step graph first: the loop capture keeps it (own slot)
                dr.dflash_capture(id_last, n_past, logits, drafts)
                dr.dflash_capture_loop(targets_d, feats_d, id_last, n_past, n_ok, logits, drafts)
                assert dr.dflash_graph_nodes(loop=True)[1] == 0
            dr.dflash_replay_loop()
        check(turn, ref_nok)
        prev_drafts = ref_drafts
    # the step graph captured before the loop graph still replays: one step at
    # the state the last loop turn left, bitwise equal to that turn's outputs
    lg, dd = logits.clone(), drafts.clone()
    logits.zero_()
    dr.dflash_replay()
    torch.cuda.synchronize()
    assert torch.equal(logits, lg) and torch.equal(drafts, dd)
    dr.close()


def test_advance_rejects_bad_sizes():
    from block_diffusion_drafter_fc_gb300 import dflash as D
    cfg = get_config("tiny_f32")
    wl = make_workload(cfg)
    dw, _ = GH.to_device(wl, "cuda")
    dr = D.Drafter(cfg, dw, max_seq=2, max_inject=16)       # room for one sequence's block only
    z = torch.zeros((2, BLOCK), dtype=torch.int32, device="cuda")
    f = torch.zeros((2, BLOCK, cfg.feat_dim), dtype=torch.float32, device="cuda")
    one = torch.zeros((2,), dtype=torch.int32, device="cuda")
    with pytest.raises(D.DFlashError, match=r"\[-3\]"):
        dr.dflash_advance(z[:, :15].contiguous(), z, f, one, one.clone(), one.clone())
    dr.close()
