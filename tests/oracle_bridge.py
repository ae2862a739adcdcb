"""Feed a synthetic workload to the fp64 oracle (test-side glue, no arithmetic)."""
from __future__ import annotations

from typing import Dict, List, Optional, Tuple

import numpy as np

from block_diffusion_drafter_fc_gb300.synth import DraftConfig, Workload, raw_numpy
from oracle import dflash_oracle as O


def oracle_config(cfg: DraftConfig) -> O.OracleConfig:
    return O.OracleConfig(
        n_layer=cfg.n_layer, n_embd=cfg.n_embd, n_head=cfg.n_head, n_head_kv=cfg.n_head_kv,
        head_dim=cfg.head_dim, n_ff=cfg.n_ff, window=cfg.window, n_vocab=cfg.n_vocab,
        weight_dtype=cfg.weight_dtype, dense_dtype=cfg.dense_dtype, ring_dtype=cfg.ring_dtype,
        rope_theta=cfg.rope_theta, eps=cfg.eps, mask_token_id=cfg.mask_token_id)


def oracle_weights(wl: Workload) -> O.OracleWeights:
    raw: Dict[str, np.ndarray] = {}
    scales: Dict[str, np.ndarray] = {}
    for name, w in wl.weights.items():
        raw[name] = raw_numpy(w.data)
        if w.scale is not None:
            scales[name] = w.scale.numpy()
    return O.OracleWeights(oracle_config(wl.cfg), raw, scales)


def oracle_prefill(wl: Workload, w: Optional[O.OracleWeights] = None,
                   calls: Optional[List[Tuple[int, int, int, int]]] = None):
    """Run the workload's inject calls through the oracle; returns (weights, rings,
    per-call H_t)."""
    w = w or oracle_weights(wl)
    rings = [O.OracleRing(w.cfg) for _ in range(wl.cfg.n_seq)]
    hts = []
    for call in (calls if calls is not None else wl.inject_calls):
        seq = call[0]
        feats = raw_numpy(wl.call_feats(call))
        H_t = O.encode(w, feats)
        O.inject(w, rings[seq], H_t, wl.positions(call).numpy())
        hts.append(H_t)
    return w, rings, hts


def oracle_full(wl: Workload, n_seq: Optional[int] = None):
    """Prefill + one block step + acceptance against the workload's synthetic
    targets built from the oracle's own drafts."""
    from block_diffusion_drafter_fc_gb300.synth import make_targets
    w, rings, hts = oracle_prefill(wl)
    n = n_seq or wl.cfg.n_seq
    logits, drafts = O.step(w, rings[:n], wl.id_last.numpy()[:n], wl.n_past.numpy()[:n])
    targets = make_targets(drafts, wl.mismatch.numpy()[:n], wl.tail.numpy()[:n], wl.cfg.n_vocab)
    n_ok = O.accept(drafts, targets)
    return dict(weights=w, rings=rings, H_t=hts, logits=logits, drafts=drafts,
                targets=targets, n_ok=n_ok)
