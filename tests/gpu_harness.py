"""Run a synthetic workload through the CUDA path via the C-ABI binding, and
compare its outputs with the oracle's (test-side glue)."""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

from block_diffusion_drafter_fc_gb300.synth import BLOCK, Workload, make_targets

# logits tolerance per storage format (max |diff| against the fp64 oracle)
LOGIT_TOL = {"f32": 1e-3, "bf16": 2e-2, "fp8": 5e-2}


def logit_tol(cfg) -> float:
    if cfg.weight_dtype == "fp8":
        return LOGIT_TOL["fp8"]
    if cfg.weight_dtype == "f32" and cfg.ring_dtype == "f32" and cfg.dense_dtype == "f32":
        return LOGIT_TOL["f32"]
    return LOGIT_TOL["bf16"]


def gpu_run(wl: Workload, n_seq: Optional[int] = None, targets: Optional[np.ndarray] = None,
            max_seq: Optional[int] = None, keep: bool = False) -> Dict:
    from block_diffusion_drafter_fc_gb300 import dflash as D
    cfg = wl.cfg
    dev = "cuda"
    dw, feats = D.to_device(wl, dev)
    max_inject = max(c[2] for c in wl.inject_calls)
    dr = D.Drafter(cfg, dw, max_seq=max_seq or cfg.n_seq, max_inject=max_inject)
    Hts = []
    for call in wl.inject_calls:
        seq, p0, cnt, r0 = call
        H = torch.empty((cnt, cfg.n_embd), dtype=torch.float32, device=dev)
        dr.dflash_encode(feats[seq][r0:r0 + cnt], H)
        pos = torch.arange(p0, p0 + cnt, dtype=torch.int32, device=dev)
        dr.dflash_inject(seq, H, pos)
        Hts.append(H)
    n = n_seq or cfg.n_seq
    id_last = wl.id_last[:n].to(dev)
    n_past = wl.n_past[:n].to(dev)
    logits = torch.empty((n, BLOCK, cfg.n_vocab), dtype=torch.float32, device=dev)
    drafts = torch.empty((n, BLOCK - 1), dtype=torch.int32, device=dev)
    dr.dflash_step(id_last, n_past, logits, drafts)
    out = dict(logits=logits.cpu().numpy(), drafts=drafts.cpu().numpy(),
               H_t=[h.cpu().numpy() for h in Hts])
    k, v, pos = dr.ring_views()
    out["ring_k"] = k.float().cpu().numpy()
    out["ring_v"] = v.float().cpu().numpy()
    out["ring_pos"] = pos.cpu().numpy()
    if targets is not None:
        t = torch.from_numpy(np.ascontiguousarray(targets)).to(dev)
        n_ok = torch.empty((n,), dtype=torch.int32, device=dev)
        dr.dflash_accept(drafts, t, n_ok)
        out["n_ok"] = n_ok.cpu().numpy()
    out["status"] = dr.dflash_read_status()
    if keep:
        out.update(drafter=dr, dev_weights=dw, feats=feats, id_last_d=id_last, n_past_d=n_past)
    else:
        dr.close()
    return out


def compare_drafts(gpu_logits, gpu_drafts, ref_logits, ref_drafts, err):
    """Drafts must equal the oracle's wherever the oracle's top-2 gap is wider
    than twice the measured logit error; inside that band (a near tie the two
    precisions may order differently) the GPU's token must be one of the
    oracle's two best.  The GPU's drafts must always be the argmax of its own
    logits (lowest index on ties).  Returns the number of positions whose token
    differs from the oracle's (0 unless a near tie flipped)."""
    own = np.argmax(gpu_logits[:, 1:, :], axis=-1)
    assert np.array_equal(own, gpu_drafts), "drafts are not the argmax of the GPU logits"
    r32 = ref_logits.astype(np.float32)[:, 1:, :]
    top2 = np.sort(r32, axis=-1)[..., -2:]
    gap = top2[..., 1] - top2[..., 0]
    clear = gap > 2 * err
    assert np.array_equal(gpu_drafts[clear], ref_drafts[clear]), "draft mismatch on a clear row"
    if (~clear).any():
        best2 = np.argsort(r32, axis=-1)[..., -2:]
        amb = np.nonzero(~clear)
        for s, j in zip(*amb):
            assert gpu_drafts[s, j] in best2[s, j], (s, j)
    # positions where the tokens actually differ (only possible inside the band)
    return int((gpu_drafts != ref_drafts).sum())


def ring_ulps(gpu_vals: np.ndarray, ref_raw: np.ndarray, dtype: str) -> np.ndarray:
    """Distance in units of the last place between two stored ring tensors."""
    if dtype == "bf16":
        a = torch.from_numpy(np.ascontiguousarray(gpu_vals.astype(np.float32))).to(torch.bfloat16)
        ai = a.view(torch.int16).numpy().astype(np.int32)
        bi = ref_raw.view(np.int16).astype(np.int32)
    else:
        ai = gpu_vals.astype(np.float32).view(np.int32).astype(np.int64)
        bi = ref_raw.astype(np.float32).view(np.int32).astype(np.int64)
    # map sign-magnitude to a monotone integer line
    ai = np.where(ai < 0, -(ai & 0x7FFFFFFF if dtype != "bf16" else ai & 0x7FFF), ai)
    bi = np.where(bi < 0, -(bi & 0x7FFFFFFF if dtype != "bf16" else bi & 0x7FFF), bi)
    return np.abs(ai - bi)
