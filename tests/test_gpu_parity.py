"""CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Bars (from the drafter's statement of the target): ring slot positions,
draft tokens and acceptance counts bit-exact; logits max |diff| <= 1e-3 with
fp32 storage, <= 2e-2 with bf16 storage, <= 5e-2 with FP8 weights.  Encoded
features H_t: max |diff| <= 1e-4 relative to their largest magnitude (fp32
math with the bf16 hi/lo activation split: ~2^-17 per product).  Ring K/V:
within one unit of the ring dtype's rounding of the oracle's value (plus
1e-5 of the tensor's scale for values near zero), since both sides round a
slightly different fp32/fp64 value once.
"""
import functools

import numpy as np
import pytest
import torch

from block_diffusion_drafter_fc_gb300.synth import (
    BLOCK, get_config, make_targets, make_workload)
import gpu_harness as GH
import oracle_bridge as OB

pytestmark = pytest.mark.gpu

SMALL = ["tiny_f32", "ragged_bf16", "mixed_f32w_bf16ring", "small_fp8", "dense_fp8", "dense_bf16",
         "wide_fp8", "wide_bf16", "many_seq_bf16", "small_fp4", "ragged_fp4", "split_bf16",
         "split_f32", "stream_h128", "stream_h64"]


@functools.lru_cache(maxsize=None)
def _case(name):
    wl = make_workload(get_config(name))
    ref = OB.oracle_full(wl)
    gpu = GH.gpu_run(wl, targets=ref["targets"])
    return wl, ref, gpu


def ring_stats(wl, ref, gpu):
    """Per sequence and K/V: positions equal, and error statistics of the stored
    values against the oracle's (in units of the tensor's max magnitude and in
    units in the last place of the ring dtype)."""
    from oracle import dflash_oracle as O
    cfg = wl.cfg
    out = []
    for s in range(cfg.n_seq):
        assert np.array_equal(gpu["ring_pos"][s], ref["rings"][s].pos), f"ring_pos seq {s}"
        filled = ref["rings"][s].pos >= 0
        for name, gk, rk in (("K", gpu["ring_k"][s], ref["rings"][s].k),
                             ("V", gpu["ring_v"][s], ref["rings"][s].v)):
            refv = O.decode(rk, cfg.ring_dtype)[:, :, filled, :]
            g = gk[:, :, filled, :].astype(np.float64)
            scale = float(np.abs(refv).max())
            d = np.abs(g - refv)
            _, e = np.frexp(np.maximum(np.abs(g), np.abs(refv)))
            ulp = np.exp2(e - (8.0 if cfg.ring_dtype == "bf16" else 24.0))
            # per element: one bf16 unit (bf16 ring), or 2^-12 of the tensor's scale.
            # The GPU value ahead of the final rounding carries the error of two
            # chained fp32-emulating projections (fc, then wk/wv: each product split
            # to 16 significant bits, ~2^-16 of the output's scale per projection),
            # and the largest of ~10^7 elements sits ~4 sigma out: 2^-12 bounds it.
            allow = np.maximum(ulp if cfg.ring_dtype == "bf16" else 0.0, 2.0 ** -12 * scale)
            out.append(dict(seq=s, name=name, max_rel_scale=float(d.max() / scale),
                            max_ulps=float((d / ulp).max()), frac_differ=float((d > 0).mean()),
                            n_bad=int((d > allow).sum()), n=int(d.size)))
    return out


def _check_ring(wl, ref, gpu):
    """bf16 ring: each stored value within one bf16 unit of the oracle's, or
    within 2^-12 of the tensor's largest magnitude (the fp32 arithmetic's error
    ahead of the final rounding, which moves values near zero by more than one
    of their own units).  fp32 ring: within 2^-12 of the tensor's scale."""
    for st in ring_stats(wl, ref, gpu):
        assert st["n_bad"] == 0, f"ring {st}"


@pytest.mark.parametrize("name", SMALL)
def test_encode_matches_oracle(name):
    wl, ref, gpu = _case(name)
    for a, b in zip(gpu["H_t"], ref["H_t"]):
        err = np.abs(a - b).max()
        assert err <= 1e-4 * np.abs(b).max(), err


@pytest.mark.parametrize("name", SMALL)
def test_ring_matches_oracle(name):
    wl, ref, gpu = _case(name)
    _check_ring(wl, ref, gpu)


@pytest.mark.parametrize("name", SMALL)
def test_step_logits_drafts_accept(name):
    wl, ref, gpu = _case(name)
    err = float(np.abs(gpu["logits"] - ref["logits"]).max())
    assert err <= GH.logit_tol(wl.cfg), err
    amb = GH.compare_drafts(gpu["logits"], gpu["drafts"], ref["logits"], ref["drafts"], err, name)
    if amb == 0:
        assert np.array_equal(gpu["drafts"], ref["drafts"])
        assert np.array_equal(gpu["n_ok"], ref["n_ok"])
    else:   # a reported near-tie flip (extra test geometries only): n_ok follows the GPU's drafts
        from oracle import dflash_oracle as O
        assert np.array_equal(gpu["n_ok"], O.accept(gpu["drafts"], ref["targets"]))
    assert gpu["status"] == 0


def test_accept_synthetic_against_oracle():
    """Accept kernel alone on synthetic drafts/targets with planted mismatches,
    including all-match (15) and mismatch at 0, for 37 sequences."""
    from block_diffusion_drafter_fc_gb300 import dflash as D
    from oracle import dflash_oracle as O
    wl = make_workload(get_config("ragged_bf16"))
    dw, _ = GH.to_device(wl)
    dr = D.Drafter(wl.cfg, dw, max_seq=37)
    g = np.random.default_rng(3)
    drafts = g.integers(0, 1000, size=(37, 15)).astype(np.int32)
    m = g.integers(0, 16, size=37)
    m[0], m[1] = 0, 15
    targets = make_targets(drafts, m, g.integers(0, 1000, size=(37, 15)), 1001)
    n_ok = torch.empty(37, dtype=torch.int32, device="cuda")
    dr.dflash_accept(torch.from_numpy(drafts).cuda(), torch.from_numpy(targets).cuda(), n_ok)
    got = n_ok.cpu().numpy()
    assert np.array_equal(got, O.accept(drafts, targets))
    assert np.array_equal(got, m)
    dr.close()


def test_fewer_sequences_than_handle():
    """n_seq = 2 on a 3-sequence handle: the first two sequences' outputs equal
    the oracle on those sequences."""
    wl = make_workload(get_config("ragged_bf16"))
    ref = OB.oracle_full(wl, n_seq=2)
    gpu = GH.gpu_run(wl, n_seq=2, targets=ref["targets"])
    bad = np.argwhere(~np.isfinite(gpu["logits"]))
    assert bad.size == 0, f"non-finite logits at (seq, row) {sorted(set(map(tuple, bad[:, :2].tolist())))}"
    err = float(np.abs(gpu["logits"] - ref["logits"]).max())
    assert err <= GH.logit_tol(wl.cfg)
    assert np.array_equal(gpu["drafts"], ref["drafts"])
    assert np.array_equal(gpu["n_ok"], ref["n_ok"])


def test_empty_ring_step():
    """A step before any injection attends only the block's own 16 keys."""
    from oracle import dflash_oracle as O
    wl = make_workload(get_config("tiny_f32"))
    w = OB.oracle_weights(wl)
    rings = [O.OracleRing(w.cfg)]
    lg, dr_ = O.step(w, rings, [int(wl.id_last[0])], [0])
    from block_diffusion_drafter_fc_gb300 import dflash as D
    dw, _ = GH.to_device(wl)
    d = D.Drafter(wl.cfg, dw)
    logits = torch.empty((1, BLOCK, wl.cfg.n_vocab), device="cuda")
    drafts = torch.empty((1, 15), dtype=torch.int32, device="cuda")
    d.dflash_step(wl.id_last[:1].cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"), logits, drafts)
    err = float(np.abs(logits.cpu().numpy() - lg).max())
    assert err <= 1e-3
    assert np.array_equal(drafts.cpu().numpy(), dr_)
    d.close()


@pytest.mark.parametrize("name", ["small_fp8", "small_fp4", "dense_bf16"])
def test_graph_replay_bitwise_with_eager_traffic(name):
    """The captured step (+accept) replays bitwise equal to the eager step, before
    and after eager GEMMs run on the same stream between replays (dflash-ops
    model card, Method: interleaved eager traffic between replays): the 16-row,
    FP4 and tcgen05 projection paths."""
    wl = make_workload(get_config(name))
    ref = OB.oracle_full(wl)
    g = GH.gpu_run(wl, targets=ref["targets"], keep=True)
    dr = g["drafter"]
    n = wl.cfg.n_seq
    logits = torch.zeros((n, BLOCK, wl.cfg.n_vocab), device="cuda")
    drafts = torch.zeros((n, 15), dtype=torch.int32, device="cuda")
    targets = torch.from_numpy(ref["targets"]).cuda()
    n_ok = torch.zeros(n, dtype=torch.int32, device="cuda")
    dr.dflash_capture(g["id_last_d"], g["n_past_d"], logits, drafts, targets, n_ok)
    a = torch.randn(2048, 2048, device="cuda", dtype=torch.bfloat16)
    outs = []
    for it in range(4):
        logits.zero_()
        drafts.zero_()
        dr.dflash_replay()
        torch.cuda.synchronize()
        outs.append((logits.clone(), drafts.clone(), n_ok.clone()))
        for _ in range(3):
            a = (a @ a).clamp_(-1, 1)
    for lg, d, k in outs:
        assert torch.equal(lg.cpu(), torch.from_numpy(g["logits"])), "replay differs from eager"
        assert np.array_equal(d.cpu().numpy(), g["drafts"])
        assert np.array_equal(k.cpu().numpy(), g["n_ok"])
    # new scalars without re-capture: a different anchor token changes the output
    g["id_last_d"].copy_((g["id_last_d"] + 1) % wl.cfg.n_vocab)
    dr.dflash_replay()
    torch.cuda.synchronize()
    assert not torch.equal(logits.cpu(), torch.from_numpy(g["logits"]))
    dr.close()


def test_step_host_matches_device_step():
    wl = make_workload(get_config("ragged_bf16"))
    g = GH.gpu_run(wl, keep=True)
    dr = g["drafter"]
    n = wl.cfg.n_seq
    drafts = torch.zeros((n, 15), dtype=torch.int32).pin_memory()
    logits = torch.zeros((n, BLOCK, wl.cfg.n_vocab), dtype=torch.float32).pin_memory()
    dr.dflash_step_host(wl.id_last.clone(), wl.n_past.clone(), drafts, logits)
    assert np.array_equal(drafts.numpy(), g["drafts"])
    assert np.array_equal(logits.numpy(), g["logits"])
    dr.close()


def test_host_side_errors_on_gpu_handle():
    from block_diffusion_drafter_fc_gb300 import dflash as D
    wl = make_workload(get_config("tiny_f32"))
    dw, feats = GH.to_device(wl)
    dr = D.Drafter(wl.cfg, dw, max_inject=80)
    H = torch.zeros((80, wl.cfg.n_embd), device="cuda")
    pos = torch.arange(80, dtype=torch.int32, device="cuda")
    with pytest.raises(D.DFlashError, match="too many rows"):
        dr.dflash_inject(0, H, pos)                      # 80 > window 64
    with pytest.raises(D.DFlashError, match="out of range"):
        dr.dflash_inject(1, H[:8], pos[:8])
    with pytest.raises(D.DFlashError, match="no captured graph"):
        dr.dflash_replay()
    ids = torch.tensor([wl.cfg.n_vocab + 5], dtype=torch.int32, device="cuda")
    lg = torch.empty((1, BLOCK, wl.cfg.n_vocab), device="cuda")
    drf = torch.empty((1, 15), dtype=torch.int32, device="cuda")
    dr.dflash_step(ids, torch.zeros(1, dtype=torch.int32, device="cuda"), lg, drf)
    assert dr.dflash_read_status() & 0x1
    assert dr.dflash_read_status() == 0                  # cleared by the read
    # zero-row encode / inject are no-ops
    dr.dflash_encode(feats[0][:0], H[:0])
    dr.dflash_inject(0, H[:0], pos[:0])
    dr.close()


@pytest.mark.slow
def test_small_bf16_full():
    wl, ref, gpu = _case("small_bf16")
    _check_ring(wl, ref, gpu)
    err = float(np.abs(gpu["logits"] - ref["logits"]).max())
    assert err <= GH.logit_tol(wl.cfg), err
    GH.compare_drafts(gpu["logits"], gpu["drafts"], ref["logits"], ref["drafts"], err, "small_bf16")
    assert np.array_equal(gpu["drafts"], ref["drafts"])
    assert np.array_equal(gpu["n_ok"], ref["n_ok"])


@pytest.mark.parametrize("name", ["tiny_f32", "ragged_bf16", "mixed_f32w_bf16ring", "split_bf16", "split_f32"])
def test_projection_chain_bitwise_equals_separate_launches(name):
    check_chain_bitwise(name)


def check_chain_bitwise(name):
    """The per-layer projection chains (o, gate/up, down, next q/k/v or the LM
    head in one launch) give the same bits as one launch per projection (the
    default), eager and replayed from a graph."""
    wl = make_workload(get_config(name))
    g = GH.gpu_run(wl, keep=True)   # one launch per projection
    dr = g["drafter"]
    n = wl.cfg.n_seq
    logits = torch.zeros((n, BLOCK, wl.cfg.n_vocab), device="cuda")
    drafts = torch.zeros((n, 15), dtype=torch.int32, device="cuda")
    dr.dflash_set_chain(True)
    dr.dflash_step(g["id_last_d"], g["n_past_d"], logits, drafts)
    torch.cuda.synchronize()
    assert np.array_equal(logits.cpu().numpy(), g["logits"])
    assert np.array_equal(drafts.cpu().numpy(), g["drafts"])
    logits.zero_()
    dr.dflash_capture(g["id_last_d"], g["n_past_d"], logits, drafts)
    assert dr.dflash_graph_nodes()[0] == 2 + 2 * wl.cfg.n_layer   # embed, q/k/v, (attention, chain) x L
    for _ in range(3):
        dr.dflash_replay()
    torch.cuda.synchronize()
    assert np.array_equal(logits.cpu().numpy(), g["logits"])
    assert dr.dflash_read_status() == 0
    dr.dflash_set_chain(False)
    dr.close()


@pytest.mark.parametrize("name", ["small_fp4", "small_fp8"])
def test_projection_chain_refused_where_unsupported(name):
    from block_diffusion_drafter_fc_gb300 import dflash as D
    wl = make_workload(get_config(name))
    dw, _ = GH.to_device(wl)
    dr = D.Drafter(wl.cfg, dw, max_seq=wl.cfg.n_seq)
    with pytest.raises(D.DFlashError, match=r"\[-2\]"):
        dr.dflash_set_chain(True)
    dr.dflash_set_chain(False)
    dr.close()


# the attention kernel each geometry's step takes (the parity cases above run
# all three)
KERNEL_OF = {"split_bf16": 0, "dense_bf16": 0, "split_f32": 0, "many_seq_bf16": 0, "stream_h128": 2,
             "stream_h64": 2}


@pytest.mark.parametrize("name", sorted(KERNEL_OF))
def test_attention_kernel_choice(name):
    wl = make_workload(get_config(name))
    g = GH.gpu_run(wl, keep=True)
    dr = g["drafter"]
    assert dr.dflash_attention_kernel(wl.cfg.n_seq) == KERNEL_OF[name]
    assert dr.dflash_attention_kernel(1) == 0
    with pytest.raises(Exception):
        dr.dflash_attention_kernel(0)
