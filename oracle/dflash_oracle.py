"""fp64 CPU oracle of the DFlash drafter block step.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
path: it reads the same stored bytes (bf16 bit patterns, f32 values, E4M3
codes with per-row f32 scales, E2M1 codes with E4M3 block and f32 row scales)
and computes the step directly from its
definition in float64, with no tiling, no online softmax and no fusion.

Sources (the documents that define the method):
  * dflash-ops model card, sections "Method", "Usage" and "Requirements and
    limits": KV injection through wk/wv with no attn_norm in front, per-head
    RMSNorm + NEOX rope on K, V stored raw, ring slot = pos mod window, the
    non-causal block attending ring (0 <= qpos - kpos < window) plus itself,
    host fp64 inverse-frequency table, greedy drafts at block rows 1..15,
    first-mismatch acceptance, fp32 arithmetic whatever the storage dtype.
  * dflash_head.rs (metrale_model_arch), struct DflashLayer and
    BlockDiffusionDraftHead fields: Qwen3-style layer (input_layernorm,
    q/k/v/o, per-head q_norm/k_norm, post_attention_layernorm, gate/up/down),
    hidden_norm and fc on the fused target context, the final norm,
    rotary_dim = head_dim, rms_norm_eps = 1e-6, and the weight-only FP8 copies
    with per-row f32 scales (enum DflashQuantization).
  * dflash_engine.py: class RMSNorm (x * rsqrt(mean(x^2) + eps) * w), class
    TargetContextFeatureFuser (H_t = RMSNorm(W_c [H^(l1); ...; H^(l5)])), class
    DFlashDraftBlock (pre-norm attention and SwiGLU MLP with residuals) and
    DFlashSpeculativeVerifier.verify_block (accepted = matching prefix length).

Readings taken where the sources are silent (each is listed in the design notes):
  * row 0 of the block sits at position n_past, row i at n_past + i;
  * a ring slot is a key for row i iff it holds a position p with 0 <= p < n_past
    and (n_past + i) - p < window; every block key is visible to every row;
  * GQA maps query head h to kv head h // (n_head / n_head_kv);
  * per-head RMSNorm comes before rope, on the block's q and k and on injected k;
  * block K/V are not written to the ring;
  * argmax ties resolve to the lowest index; the greedy decision is taken on the
    logits rounded to fp32, the precision the model card fixes for the arithmetic;
  * ring values are the fp64 results rounded once (nearest-even) to the ring dtype.

Every function here is pinned by the CPU tests against closed forms,
library routines (torch float64 SDPA / rms_norm / silu, torch dtype casts),
brute force on tiny inputs, the verifier example printed in dflash_engine.py,
and the structural invariants the model card lists (ring wraparound, window
masking by perturbing out-of-window slots, non-causal joint denoising,
determinism, relative-position invariance of rope).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np

BLOCK = 16


# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64.  A bf16 value is the upper half of
    the IEEE binary32 with the same bits."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 to the nearest bf16 (ties to even) and return its bits.

    bf16 keeps 8 significant bits and binary32's exponent range, so the quantum
    of a normal |x| in [2^(e-1), 2^e) is 2^(e-8); below 2^-126 the quantum is the
    subnormal step 2^-133.  The rounded value is exact in binary32, whose upper
    16 bits are the bf16 pattern."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.exp2(np.maximum(e.astype(np.float64) - 8.0, -133.0))
    r = np.rint(x / q) * q                      # np.rint rounds half to even
    with np.errstate(over="ignore"):
        f = r.astype(np.float32)
    f = np.where(np.abs(r) > 3.3895313892515355e38, np.copysign(np.inf, r), f).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """FP8 E4M3 (fn variant: bias 7, no infinities, S.1111.111 = NaN) -> float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    v = s * np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, v)


def e2m1_to_f64(codes: np.ndarray) -> np.ndarray:
    """FP4 E2M1 codes (4 bits: sign, 2 exponent bits with bias 1, 1 mantissa bit;
    no infinities or NaN) -> float64: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives."""
    c = np.asarray(codes, dtype=np.int64) & 0xF
    s = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    return s * np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e - 1.0))


def decode(raw: np.ndarray, dtype: str, scale: Optional[np.ndarray] = None) -> np.ndarray:
    """Stored tensor -> float64 values.  FP8 rows are multiplied by their f32
    scale: y[n] = s[n] * sum_k q[n,k] x[k] is the same as using s[n] * q[n,k].
    FP4 (the self-defined block-scaled format of the weights) is one flat byte
    buffer per [N, K] matrix, N = len(scale): w[n,k] = s[n] *
    e4m3(block[n, k // 16]) * e2m1(code[n,k]).  The first N K/2 bytes are the
    codes, row-major; within each 16-byte group of a row (32 weights) byte
    4t + j holds the codes of k = 2 (t + 4j) (low nibble) and k + 1 (high
    nibble), t, j = 0..3.  Then ceil(N/16) x K/16 blocks of 16 scale bytes:
    block b of row group G holds block b's scales of rows 16G + (0, 8, 1, 9,
    ..., 7, 15)."""
    if dtype == "bf16":
        return bf16_to_f64(raw)
    if dtype == "f32":
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    if dtype == "fp8":
        v = e4m3_to_f64(raw)
        return v * np.asarray(scale, dtype=np.float64)[:, None]
    if dtype == "fp4":
        r = np.asarray(raw, dtype=np.uint8).reshape(-1)
        n = len(scale)
        groups = -(-n // 16)
        k = 2 * r.size // (n + 2 * groups)          # size = n k/2 + groups 16 k/16
        codes = r[:n * k // 2].reshape(n, k // 2)
        # stored byte 4t + j of a group -> code pair t + 4j (the 4 x 4 transpose)
        codes = codes.reshape(n, k // 32, 4, 4).transpose(0, 1, 3, 2).reshape(n, k // 2)
        # scale byte p of block (G, b) -> row 16G + p // 2 + 8 (p % 2)
        sb = r[n * k // 2:].reshape(groups, k // 16, 16)
        p = np.arange(16)
        blocks = np.empty((groups * 16, k // 16), dtype=np.uint8)
        blocks[(np.arange(groups)[:, None] * 16 + p // 2 + 8 * (p % 2)).reshape(-1)] = \
            sb.transpose(0, 2, 1).reshape(groups * 16, k // 16)
        blocks = blocks[:n]
        v = np.empty((n, k), dtype=np.float64)
        v[:, 0::2] = e2m1_to_f64(codes & 0xF)
        v[:, 1::2] = e2m1_to_f64(codes >> 4)
        v *= np.repeat(e4m3_to_f64(blocks), 16, axis=1)
        return v * np.asarray(scale, dtype=np.float64)[:, None]
    raise ValueError(dtype)


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once to a ring storage dtype (raw form)."""
    if dtype == "bf16":
        return f64_to_bf16(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# the drafter's building blocks
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w over the last axis (dflash_engine.py, class
    RMSNorm; eps 1e-6 as in dflash_head.rs, field rms_norm_eps)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def inv_freq_table(theta: float, head_dim: int) -> np.ndarray:
    """inv_freq[j] = theta^(-2j/head_dim), j < head_dim/2, in float64 (dflash-ops
    model card, Method: a host fp64 inverse-frequency table; rotary_dim = head_dim
    per dflash_head.rs, field rotary_dim)."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * j / head_dim)


def rope_neox(x: np.ndarray, pos: np.ndarray, inv_freq: np.ndarray) -> np.ndarray:
    """NEOX rotary embedding over the whole head: element j pairs with j + hd/2.
    x[..., hd] at integer positions pos[...] (broadcast over the middle axes)."""
    half = x.shape[-1] // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq       # [..., half]
    while ang.ndim < x.ndim:
        ang = ang[..., None, :]                                          # broadcast heads
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T for a row-major weight W[out, in]."""
    return x @ w.T


# ---------------------------------------------------------------------------
# model containers
# ---------------------------------------------------------------------------

@dataclass
class OracleConfig:
    n_layer: int
    n_embd: int
    n_head: int
    n_head_kv: int
    head_dim: int
    n_ff: int
    window: int
    n_vocab: int
    weight_dtype: str
    dense_dtype: str
    ring_dtype: str
    rope_theta: float
    eps: float
    mask_token_id: int


class OracleWeights:
    """Stored weights decoded lazily to float64 (one matrix at a time, so the
    real-dimension configurations fit in host memory)."""

    def __init__(self, cfg: OracleConfig, raw: Dict[str, np.ndarray],
                 scales: Optional[Dict[str, np.ndarray]] = None):
        self.cfg = cfg
        self.raw = raw
        self.scales = scales or {}

    def dtype_of(self, name: str) -> str:
        base = name.split(".")[-1]
        if base in ("wq", "wk", "wv", "wo", "gate", "up", "down") or name == "lm_head":
            return self.cfg.weight_dtype
        return self.cfg.dense_dtype

    def get(self, name: str) -> np.ndarray:
        return decode(self.raw[name], self.dtype_of(name), self.scales.get(name))

    def rows(self, name: str, idx: np.ndarray) -> np.ndarray:
        """Selected rows of a dense matrix (the embedding gather)."""
        return decode(np.asarray(self.raw[name])[idx], self.dtype_of(name))


class OracleRing:
    """One sequence's sliding-window ring: K and V per layer in the ring's storage
    dtype, [L][n_head_kv][window][head_dim], and the position each slot holds
    (-1 = empty), shared by every layer."""

    def __init__(self, cfg: OracleConfig):
        shp = (cfg.n_layer, cfg.n_head_kv, cfg.window, cfg.head_dim)
        dt = np.uint16 if cfg.ring_dtype == "bf16" else np.float32
        self.cfg = cfg
        self.k = np.zeros(shp, dtype=dt)
        self.v = np.zeros(shp, dtype=dt)
        self.pos = np.full((cfg.window,), -1, dtype=np.int64)

    def copy(self) -> "OracleRing":
        r = OracleRing(self.cfg)
        r.k, r.v, r.pos = self.k.copy(), self.v.copy(), self.pos.copy()
        return r

    def values(self, layer: int):
        d = self.cfg.ring_dtype
        return decode(self.k[layer], d), decode(self.v[layer], d)


# ---------------------------------------------------------------------------
# encode + inject (the target-feature side)
# ---------------------------------------------------------------------------

def encode(w: OracleWeights, feats: np.ndarray) -> np.ndarray:
    """H_t = RMSNorm(feats fc^T) * hidden_norm (dflash_engine.py, class
    TargetContextFeatureFuser; dflash_head.rs fields fc and hidden_norm).
    feats: stored [T, n_target_layers * d_target] -> float64 [T, n_embd]."""
    cfg = w.cfg
    f = decode(feats, cfg.dense_dtype)
    return rmsnorm(linear(f, w.get("fc")), w.get("hidden_norm"), cfg.eps)


def inject_kv(w: OracleWeights, layer: int, H_t: np.ndarray, positions: np.ndarray,
              inv_freq: np.ndarray):
    """One layer's context K/V from fused features, before storage rounding:
    K = rope(RMSNorm_head(H_t wk^T) * k_norm, pos), V = H_t wv^T; no attn_norm in
    front (dflash-ops model card, Method)."""
    cfg = w.cfg
    T = H_t.shape[0]
    k = linear(H_t, w.get(f"l{layer}.wk")).reshape(T, cfg.n_head_kv, cfg.head_dim)
    k = rmsnorm(k, w.get(f"l{layer}.k_norm"), cfg.eps)
    k = rope_neox(k, positions, inv_freq)
    v = linear(H_t, w.get(f"l{layer}.wv")).reshape(T, cfg.n_head_kv, cfg.head_dim)
    return k, v


def inject(w: OracleWeights, ring: OracleRing, H_t: np.ndarray, positions: Sequence[int]) -> None:
    """Write every layer's K/V of the given rows into slot pos mod window, in row
    order, and record the slot's position (dflash-ops model card, Usage and
    Requirements: slots are pos % window, later writes overwrite earlier ones,
    at most `window` rows per call)."""
    cfg = w.cfg
    positions = np.asarray(positions, dtype=np.int64)
    assert H_t.shape[0] == positions.shape[0] <= cfg.window
    inv_freq = inv_freq_table(cfg.rope_theta, cfg.head_dim)
    for layer in range(cfg.n_layer):
        k, v = inject_kv(w, layer, H_t, positions, inv_freq)
        ks, vs = store(k, cfg.ring_dtype), store(v, cfg.ring_dtype)
        for t, p in enumerate(positions):
            slot = int(p) % cfg.window
            ring.k[layer, :, slot, :] = ks[t]
            ring.v[layer, :, slot, :] = vs[t]
    for p in positions:
        ring.pos[int(p) % cfg.window] = int(p)


# ---------------------------------------------------------------------------
# the block step
# ---------------------------------------------------------------------------

def ring_mask(ring_pos: np.ndarray, n_past: int, window: int, rows: int = BLOCK) -> np.ndarray:
    """valid[i, s] for block row i (position n_past + i, i < rows) and ring slot
    s: the slot holds a past position p (0 <= p < n_past) within the window,
    (n_past + i) - p < window (dflash-ops model card, Method)."""
    p = np.asarray(ring_pos, dtype=np.int64)[None, :]
    q = n_past + np.arange(rows, dtype=np.int64)[:, None]
    return (p >= 0) & (p < n_past) & (q - p < window)


def attention(q: np.ndarray, k_blk: np.ndarray, v_blk: np.ndarray,
              k_ring: np.ndarray, v_ring: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """Non-causal sliding-window GQA attention of one sequence's block.
    q [16, Hq, hd]; k_blk, v_blk [16, Hkv, hd]; k_ring, v_ring [Hkv, W, hd];
    valid [16, W].  Keys = the valid ring slots plus all 16 block rows; scores
    scaled by 1/sqrt(hd); exact softmax.  Returns [16, Hq, hd]."""
    n_q, hq, hd = q.shape
    hkv = k_blk.shape[1]
    group = hq // hkv
    out = np.zeros_like(q)
    scale = 1.0 / np.sqrt(hd)
    for h in range(hq):
        g = h // group
        keys = np.concatenate([k_ring[g], k_blk[:, g, :]], axis=0)      # [W+16, hd]
        vals = np.concatenate([v_ring[g], v_blk[:, g, :]], axis=0)
        s = (q[:, h, :] @ keys.T) * scale                                # [16, W+16]
        mask = np.concatenate([valid, np.ones((n_q, k_blk.shape[0]), dtype=bool)], axis=1)
        s = np.where(mask, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vals
    return out


def block_tokens(cfg: OracleConfig, id_last: int, width: int = BLOCK) -> np.ndarray:
    """[id_last, mask x (width - 1)]: the anchor then the mask tokens (dflash-ops
    model card, Method; dflash_head.rs field mask_token_id).  The block holds
    width rows: 16 by default, or the scheduler's narrower block_g
    (dflash_head.rs, set_block_g: the anchor plus num_drafts mask rows)."""
    t = np.full((width,), cfg.mask_token_id, dtype=np.int64)
    t[0] = id_last
    return t


def step_hidden(w: OracleWeights, rings: List[OracleRing], tokens: np.ndarray,
                n_past: Sequence[int], causal: bool = False) -> np.ndarray:
    """Final hidden state (before the output norm) of every block row.
    tokens [n_seq, B] (B = block width, 16 by default); returns float64
    [n_seq, B, n_embd].  `causal=True` is a comparison variant used only by the
    tests (block keys j <= i)."""
    cfg = w.cfg
    n_seq, B = tokens.shape
    inv_freq = inv_freq_table(cfg.rope_theta, cfg.head_dim)
    hd, hq, hkv = cfg.head_dim, cfg.n_head, cfg.n_head_kv
    h = w.rows("tok_embd", tokens.reshape(-1)).reshape(n_seq, B, cfg.n_embd)
    pos = np.asarray(n_past, dtype=np.int64)[:, None] + np.arange(B)[None, :]
    for layer in range(cfg.n_layer):
        L = f"l{layer}."
        x = rmsnorm(h, w.get(L + "attn_norm"), cfg.eps)
        q = linear(x, w.get(L + "wq")).reshape(n_seq, B, hq, hd)
        k = linear(x, w.get(L + "wk")).reshape(n_seq, B, hkv, hd)
        v = linear(x, w.get(L + "wv")).reshape(n_seq, B, hkv, hd)
        q = rope_neox(rmsnorm(q, w.get(L + "q_norm"), cfg.eps), pos, inv_freq)
        k = rope_neox(rmsnorm(k, w.get(L + "k_norm"), cfg.eps), pos, inv_freq)
        att = np.zeros((n_seq, B, hq, hd))
        for s in range(n_seq):
            kr, vr = rings[s].values(layer)
            valid = ring_mask(rings[s].pos, int(n_past[s]), cfg.window, B)
            if causal:
                att[s] = _causal_attention(q[s], k[s], v[s], kr, vr, valid)
            else:
                att[s] = attention(q[s], k[s], v[s], kr, vr, valid)
        h = h + linear(att.reshape(n_seq, B, hq * hd), w.get(L + "wo"))
        x2 = rmsnorm(h, w.get(L + "ffn_norm"), cfg.eps)
        mlp = silu(linear(x2, w.get(L + "gate"))) * linear(x2, w.get(L + "up"))
        h = h + linear(mlp, w.get(L + "down"))
    return h


def logits_from_hidden(w: OracleWeights, h: np.ndarray) -> np.ndarray:
    """logits = RMSNorm(h) * out_norm lm_head^T for all 16 rows (dflash-ops model
    card, Usage: step returns [16, n_vocab]; lm_head borrowed from the target)."""
    cfg = w.cfg
    return linear(rmsnorm(h, w.get("out_norm"), cfg.eps), w.get("lm_head"))


def greedy_drafts(logits: np.ndarray) -> np.ndarray:
    """drafts[j] = argmax of block row j + 1 (rows 1..15; row 0 unused), decided on
    the logits rounded to fp32; ties go to the lowest index (np.argmax)."""
    l32 = np.asarray(logits, dtype=np.float64).astype(np.float32)
    return np.argmax(l32[..., 1:, :], axis=-1).astype(np.int32)


def step(w: OracleWeights, rings: List[OracleRing], id_last: Sequence[int],
         n_past: Sequence[int], width: int = BLOCK):
    """One block step of `width` rows for n_seq sequences: (logits float64
    [n_seq, width, V], drafts int32 [n_seq, width - 1])."""
    tokens = np.stack([block_tokens(w.cfg, int(t), width) for t in id_last])
    h = step_hidden(w, rings, tokens, n_past)
    logits = logits_from_hidden(w, h)
    return logits, greedy_drafts(logits)


def accept(drafts: np.ndarray, targets: np.ndarray) -> np.ndarray:
    """n_ok per sequence = length of the prefix where drafts equal the target's
    tokens (dflash_engine.py, DFlashSpeculativeVerifier.verify_block; 15 when all
    agree).  The bonus token is not part of this count."""
    drafts = np.asarray(drafts)
    targets = np.asarray(targets)
    out = np.zeros((drafts.shape[0],), dtype=np.int32)
    for s in range(drafts.shape[0]):
        n = 0
        while n < drafts.shape[1] and drafts[s, n] == targets[s, n]:
            n += 1
        out[s] = n
    return out


def advance(w: OracleWeights, rings: List[OracleRing], drafts: np.ndarray, targets: np.ndarray,
            feats: np.ndarray, id_last: Sequence[int], n_past: Sequence[int]):
    """One turn of the speculative loop after the target has verified the drafted
    block (dflash_engine.py, DFlashSpeculativeVerifier.verify_block: the accepted
    drafts plus one token of the target; dflash-ops model card, Usage: the target's
    features of the verified positions are encoded and injected before the next
    step(id_last, n_past)).

    targets[s] holds the target's token at each block row (row j predicts
    position n_past + j + 1) and feats[s] its features at the block rows; drafts
    has one column per drafted row (15 for a 16-row block).  With
    m = accept(drafts, targets[:, :drafts.shape[1]])[s]: block rows 0..m (positions
    n_past .. n_past + m) are the verified context and are injected; the next
    anchor is the target's token m; n_past grows by m + 1.  Rings change in place;
    returns (n_ok, id_last, n_past) as new arrays."""
    targets = np.asarray(targets)
    n_ok = accept(drafts, targets[:, :np.asarray(drafts).shape[1]])
    new_id = np.zeros((len(rings),), dtype=np.int32)
    new_np = np.zeros((len(rings),), dtype=np.int32)
    for s, ring in enumerate(rings):
        m = int(n_ok[s])
        p0 = int(n_past[s])
        H_t = encode(w, np.asarray(feats[s])[:m + 1])
        inject(w, ring, H_t, np.arange(p0, p0 + m + 1))
        new_id[s] = targets[s, m]
        new_np[s] = p0 + m + 1
    return n_ok, new_id, new_np


def _causal_attention(q, k_blk, v_blk, k_ring, v_ring, valid):
    """Comparison variant for the non-causality pin: block key j visible to row i
    only when j <= i.  Not part of the method."""
    n_q, hq, hd = q.shape
    hkv = k_blk.shape[1]
    out = np.zeros_like(q)
    scale = 1.0 / np.sqrt(hd)
    tri = np.tril(np.ones((n_q, n_q), dtype=bool))
    for h in range(hq):
        g = h // (hq // hkv)
        keys = np.concatenate([k_ring[g], k_blk[:, g, :]], axis=0)
        vals = np.concatenate([v_ring[g], v_blk[:, g, :]], axis=0)
        s = (q[:, h, :] @ keys.T) * scale
        s = np.where(np.concatenate([valid, tri], axis=1), s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        out[:, h, :] = (p / p.sum(axis=1, keepdims=True)) @ vals
    return out
