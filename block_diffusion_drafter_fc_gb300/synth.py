"""Seeded synthetic workloads for the DFlash drafter block step.

This module only draws numbers and lays them out; it holds none of the
drafter's arithmetic.  Both the CUDA path and the fp64 oracle consume the
exact bytes produced here (weights rounded once to their storage dtype,
features, token ids, positions, mismatch indices).

Shapes follow the workloads described on the dflash-ops model card
(section "Measured": 5 layers, n_embd 6656, 32/8 heads of 128, n_ff 19968,
window 2048, block 16, vocabulary 8192) and the cross-sequence batch of
dflash_head.rs (struct DflashBatch, enum DflashQuantization).  No trained
weights exist here, so every tensor is random: weights ~ N(0, 1/fan_in),
norm weights 1 + N(0, 0.02), features ~ N(0, 1), token embeddings ~ N(0, 1).

FP8 weights are made the way dflash_head.rs describes its weight-only FP8
copies: one f32 scale per output row, s[n] = max_k |w[n,k]| / 448, and the
stored byte is the E4M3 (fn variant) code of w[n,k] / s[n], rounded to
nearest-even and clamped to +-448.  That is weight preparation, not a step
of the drafter; the cast itself is torch's float8_e4m3fn conversion.

FP4 weights (dflash_head.rs names an NVFP4 LM head; its layout is not on the
pages, so the format here is self-defined in the same spirit): an E2M1 code
per weight (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives), one E4M3
block scale per 16 consecutive weights of a row and one f32 scale per row:
w = s_row * e4m3(block) * e2m1(code).  s_row = max |w_row| / (6 * 448); the
block scale is the E4M3 rounding of max |w_block| / (6 s_row); codes are the
nearest E2M1 values of w / (s_row * block) (ties to the even code, +-6 at
most).  Stored per matrix as one byte buffer: N x K/2 code bytes, then the
block scales of each group of 16 rows.  Codes: row-major; within each 16-byte
group of a row (32 weights) byte 4t + j holds the codes of k = 2 (t + 4j) (low
nibble) and k + 1 (high nibble), t, j = 0..3, so the four bytes one lane of the
16-row kernel's MMA fragment needs for two k16 steps sit in one word.  Scales:
ceil(N/16) x K/16 blocks of 16 bytes; block b of row group G holds the scales of
block b of rows 16G + (0, 8, 1, 9, ..., 7, 15) (rows past N are zero), so a
lane reads the scales of rows g and g + 8 as one 16-bit pair and the 16 rows x
256 k of one pipeline stage are 256 contiguous bytes.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

BLOCK = 16          # tokens in one noise block (anchor + 15 masks)
FP8_MAX = 448.0     # largest finite E4M3 (fn) magnitude

DTYPES = ("f32", "bf16", "fp8", "fp4")
FP4_MAX = 6.0       # largest E2M1 magnitude
FP4_BLOCK = 16      # weights per E4M3 block scale
_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class DraftConfig:
    """Drafter geometry, storage formats and the synthetic workload recipe."""

    name: str
    n_layer: int
    n_embd: int
    n_head: int
    n_head_kv: int
    head_dim: int
    n_ff: int
    window: int
    n_vocab: int
    weight_dtype: str           # q/k/v/o/gate/up/down and lm_head: f32 | bf16 | fp8 | fp4
    dense_dtype: str            # tok_embd, fc, norm weights, target features: f32 | bf16
    ring_dtype: str             # ring K/V: f32 | bf16
    n_seq: int = 1
    n_target_layers: int = 5
    target_embd: int = 0        # 0 -> n_embd
    rope_theta: float = 1e6
    eps: float = 1e-6
    # inject schedule for one-sequence workloads: list of (first_pos, count)
    inject: Tuple[Tuple[int, int], ...] = ()
    # batched workloads: fill ~ U{fill_lo..fill_hi}, offset ~ U{0..offset_hi}
    fill_lo: int = 0
    fill_hi: int = 0
    offset_hi: int = 0
    mismatch: str = "uniform"   # uniform in 0..15 | geometric(p) capped at 15
    mismatch_p: float = 0.35
    seed: int = 1000

    @property
    def d_t(self) -> int:
        return self.target_embd or self.n_embd

    @property
    def feat_dim(self) -> int:
        return self.n_target_layers * self.d_t

    @property
    def qd(self) -> int:
        return self.n_head * self.head_dim

    @property
    def kvd(self) -> int:
        return self.n_head_kv * self.head_dim

    @property
    def mask_token_id(self) -> int:
        return self.n_vocab - 1

    def weight_params(self) -> int:
        """Parameters of the GEMM weights streamed by one block step."""
        per_layer = (self.qd + 2 * self.kvd) * self.n_embd + self.n_embd * self.qd \
            + 3 * self.n_ff * self.n_embd
        return self.n_layer * per_layer + self.n_vocab * self.n_embd

    def with_(self, **kw) -> "DraftConfig":
        return dataclasses.replace(self, **kw)


def _cfg_list() -> List[DraftConfig]:
    tiny = DraftConfig(
        name="tiny_f32", n_layer=1, n_embd=256, n_head=4, n_head_kv=2, head_dim=64,
        n_ff=768, window=64, n_vocab=512, weight_dtype="f32", dense_dtype="f32",
        ring_dtype="f32", inject=((0, 64), (64, 16)), seed=1000)
    small = DraftConfig(
        name="small_bf16", n_layer=3, n_embd=2048, n_head=16, n_head_kv=4, head_dim=128,
        n_ff=6144, window=512, n_vocab=32000, weight_dtype="bf16", dense_dtype="bf16",
        ring_dtype="bf16", inject=((0, 512), (512, 37)), seed=1001)
    real_bf16 = DraftConfig(
        name="real_bf16", n_layer=5, n_embd=6656, n_head=32, n_head_kv=8, head_dim=128,
        n_ff=19968, window=2048, n_vocab=8192, weight_dtype="bf16", dense_dtype="bf16",
        ring_dtype="bf16", inject=((0, 2048),), seed=1002)
    real_f32 = real_bf16.with_(name="real_f32", weight_dtype="f32", dense_dtype="f32",
                               ring_dtype="f32", seed=1003)
    batched_fp8 = DraftConfig(
        name="batched_fp8", n_layer=5, n_embd=4096, n_head=32, n_head_kv=8, head_dim=128,
        n_ff=12288, window=2048, n_vocab=32768, weight_dtype="fp8", dense_dtype="bf16",
        ring_dtype="bf16", n_seq=32, fill_lo=256, fill_hi=2048, offset_hi=65535,
        mismatch="geometric", mismatch_p=0.35, seed=1004)
    # the real-dimension drafter with FP4 projection weights (the quantized drafter
    # of the dflash-ops model card, Measured: a ~4.6-bit drafter; here 4.5 bits a
    # weight + one f32 per row)
    real_fp4 = real_bf16.with_(name="real_fp4", weight_dtype="fp4", seed=1005)
    # ... and with E4M3 projection weights (one sequence: the 16-row E4M3 path)
    real_fp8 = real_bf16.with_(name="real_fp8", weight_dtype="fp8", seed=1006)
    return [tiny, small, real_bf16, real_f32, batched_fp8, real_fp4, real_fp8]


CONFIGS: List[DraftConfig] = _cfg_list()
BY_NAME: Dict[str, DraftConfig] = {c.name: c for c in CONFIGS}

# Test-only geometries: ragged vocab / n_ff / row counts, several sequences,
# and a batched FP8 case small enough for the oracle to finish in seconds.
RAGGED = DraftConfig(
    name="ragged_bf16", n_layer=2, n_embd=320, n_head=5, n_head_kv=1, head_dim=64,
    n_ff=800, window=48, n_vocab=1001, weight_dtype="bf16", dense_dtype="bf16",
    ring_dtype="bf16", n_seq=3, fill_lo=20, fill_hi=48, offset_hi=300, seed=2001)
SMALL_FP8 = DraftConfig(
    name="small_fp8", n_layer=2, n_embd=512, n_head=8, n_head_kv=2, head_dim=64,
    n_ff=1536, window=128, n_vocab=3000, weight_dtype="fp8", dense_dtype="bf16",
    ring_dtype="bf16", n_seq=5, fill_lo=32, fill_hi=128, offset_hi=65535,
    mismatch="geometric", seed=2002)
MIXED_F32 = DraftConfig(
    name="mixed_f32w_bf16ring", n_layer=2, n_embd=256, n_head=4, n_head_kv=4, head_dim=64,
    n_ff=544, window=40, n_vocab=777, weight_dtype="f32", dense_dtype="f32",
    ring_dtype="bf16", n_seq=2, fill_lo=8, fill_hi=40, offset_hi=1000, seed=2003)
# batches of >= 128 block rows (the tcgen05 projection path): a ragged last
# 128-row tile with FP8 weights, and bf16 weights
DENSE_FP8 = SMALL_FP8.with_(name="dense_fp8", n_seq=9, seed=2004)
DENSE_BF16 = SMALL_FP8.with_(name="dense_bf16", n_seq=8, weight_dtype="bf16", mismatch="uniform",
                             seed=2005)
# wide gate/up and LM head (> 2 x 152 n-tiles of 128 rows): the tcgen05 path's
# 256-row weight tiles, FP8 with a ragged row tile and bf16
WIDE_FP8 = SMALL_FP8.with_(name="wide_fp8", n_layer=1, n_embd=256, n_head=4, n_head_kv=2,
                           n_ff=20480, n_vocab=40000, n_seq=9, seed=2006)
WIDE_BF16 = WIDE_FP8.with_(name="wide_bf16", weight_dtype="bf16", mismatch="uniform", n_seq=8,
                           seed=2007)
# enough sequences that attention gives every CTA a whole window (no cluster
# split: > 2 x 152 CTAs without one)
MANY_SEQ = DraftConfig(
    name="many_seq_bf16", n_layer=1, n_embd=256, n_head=8, n_head_kv=4, head_dim=64,
    n_ff=512, window=128, n_vocab=512, weight_dtype="bf16", dense_dtype="bf16",
    ring_dtype="bf16", n_seq=80, fill_lo=16, fill_hi=128, offset_hi=4000, seed=2008)
# FP4 weights: K (n_embd, qd, n_ff) multiples of 256, several sequences
SMALL_FP4 = DraftConfig(
    name="small_fp4", n_layer=2, n_embd=512, n_head=8, n_head_kv=2, head_dim=64,
    n_ff=1536, window=128, n_vocab=3000, weight_dtype="fp4", dense_dtype="bf16",
    ring_dtype="bf16", n_seq=3, fill_lo=32, fill_hi=128, offset_hi=65535, seed=2009)
# FP4 with head_dim 32 and one kv head: the k and v segments (32 rows each) do
# not fill 64-row boxes, the vocabulary leaves a ragged last tile
RAGGED_FP4 = DraftConfig(
    name="ragged_fp4", n_layer=1, n_embd=256, n_head=8, n_head_kv=1, head_dim=32,
    n_ff=512, window=64, n_vocab=333, weight_dtype="fp4", dense_dtype="bf16",
    ring_dtype="bf16", n_seq=2, fill_lo=20, fill_hi=64, offset_hi=500, seed=2010)
# windows of several 128-slot attention splits: a ragged last split, partly
# filled and wrapped rings (bf16, two query heads per kv head), and an fp32 ring
# with head_dim 128 and four query heads per kv head, injected past the window
SPLIT_BF16 = DraftConfig(
    name="split_bf16", n_layer=1, n_embd=256, n_head=4, n_head_kv=2, head_dim=64,
    n_ff=512, window=448, n_vocab=700, weight_dtype="bf16", dense_dtype="bf16",
    ring_dtype="bf16", n_seq=2, fill_lo=100, fill_hi=448, offset_hi=3000, seed=2011)
SPLIT_F32 = DraftConfig(
    name="split_f32", n_layer=1, n_embd=512, n_head=8, n_head_kv=2, head_dim=128,
    n_ff=512, window=320, n_vocab=600, weight_dtype="f32", dense_dtype="f32",
    ring_dtype="f32", inject=((0, 320), (320, 50)), seed=2012)
# batches whose split grid exceeds one wave (stream-K attention): windows cut
# across CTAs and merged, head_dim 128 with four query heads per kv head, and
# head_dim 64 with a window that ends inside a 64-slot sub-chunk
STREAM_H128 = DraftConfig(
    name="stream_h128", n_layer=1, n_embd=512, n_head=8, n_head_kv=2, head_dim=128,
    n_ff=512, window=576, n_vocab=600, weight_dtype="bf16", dense_dtype="bf16",
    ring_dtype="bf16", n_seq=24, fill_lo=40, fill_hi=576, offset_hi=5000, seed=2013)
STREAM_H64 = DraftConfig(
    name="stream_h64", n_layer=2, n_embd=256, n_head=4, n_head_kv=2, head_dim=64,
    n_ff=512, window=456, n_vocab=500, weight_dtype="bf16", dense_dtype="bf16",
    ring_dtype="bf16", n_seq=72, fill_lo=10, fill_hi=456, offset_hi=3000, seed=2014)
TEST_CONFIGS: Dict[str, DraftConfig] = {c.name: c for c in (RAGGED, SMALL_FP8, MIXED_F32, DENSE_FP8,
                                                            DENSE_BF16, WIDE_FP8, WIDE_BF16, MANY_SEQ,
                                                            SMALL_FP4, RAGGED_FP4, SPLIT_BF16,
                                                            SPLIT_F32, STREAM_H128, STREAM_H64)}


def get_config(name: str) -> DraftConfig:
    if name in BY_NAME:
        return BY_NAME[name]
    return TEST_CONFIGS[name]


# --------------------------------------------------------------------------
# storage helpers (no drafter arithmetic: rounding a draw to its format)
# --------------------------------------------------------------------------

def _store_dense(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(_TORCH[dtype]).contiguous()


def quantize_fp8_rows(w: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-row FP8 E4M3 copy of a f32 matrix: (codes uint8 [N,K], scales f32 [N]),
    computed in row blocks on the thread pool."""
    n_rows = w.shape[0]
    q = torch.empty(w.shape, dtype=torch.uint8)
    s = torch.empty(n_rows, dtype=torch.float32)
    step = max(1, _CHUNK // max(1, w.shape[1]))

    def blk(r0):
        x = w[r0:r0 + step]
        amax = x.abs().amax(dim=1)
        sc = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax)).to(torch.float32)
        s[r0:r0 + step] = sc
        q[r0:r0 + step] = (x / sc[:, None]).clamp_(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn).view(torch.uint8)

    list(_POOL.map(blk, range(0, n_rows, step)))
    return q, s


# E2M1 magnitudes by code (bit 3 is the sign) and the rounding boundaries
# between neighbours: a tie rounds to the code with an even mantissa bit
_E2M1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_codes(y: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code (4 bits) of each value, ties to the even code, +-6 at most."""
    a = y.abs().clamp(max=FP4_MAX)
    # magnitude code = number of grid points below the value's rounding interval
    mids = (_E2M1[1:] + _E2M1[:-1]) / 2            # 0.25 0.75 1.25 1.75 2.5 3.5 5
    idx = torch.bucketize(a, mids, right=False)     # a <= mid -> lower point
    # at an exact midpoint bucketize chose the lower point: keep it when that code is
    # even, else take the upper one
    tie = (idx < 7) & (a == mids[idx.clamp(max=6)]) & (idx % 2 == 1)
    idx = idx + tie.to(idx.dtype)
    return (idx | ((y < 0) & (idx > 0)).to(idx.dtype) << 3).to(torch.uint8)


def fp4_nbytes(n_rows: int, k: int) -> int:
    """Size of the FP4 byte buffer of an [N, K] matrix: codes + padded block scales."""
    return n_rows * k // 2 + -(-n_rows // 16) * 16 * (k // FP4_BLOCK)


def quantize_fp4_rows(w: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """FP4 copy of a f32 matrix [N, K] (K % 32 == 0): (bytes uint8 [fp4_nbytes]
    = codes then block scales, row scales f32 [N]), in row blocks on the pool."""
    n_rows, k = w.shape
    nb = k // FP4_BLOCK
    codes = torch.empty((n_rows, k // 2), dtype=torch.uint8)
    bsc = torch.empty((n_rows, nb), dtype=torch.uint8)
    s = torch.empty(n_rows, dtype=torch.float32)
    step = max(1, _CHUNK // max(1, k))

    def blk(r0):
        x = w[r0:r0 + step]
        amax = x.abs().amax(dim=1)
        sr = torch.where(amax > 0, amax / (FP4_MAX * FP8_MAX), torch.ones_like(amax)).to(torch.float32)
        s[r0:r0 + step] = sr
        xb = x.view(x.shape[0], nb, FP4_BLOCK)
        bmax = xb.abs().amax(dim=2)
        b8 = (bmax / (FP4_MAX * sr[:, None])).clamp_(max=FP8_MAX).to(torch.float8_e4m3fn)
        bsc[r0:r0 + step] = b8.view(torch.uint8)
        b = b8.to(torch.float32)
        denom = (b * sr[:, None])[:, :, None]
        y = torch.where(denom > 0, xb / torch.where(denom > 0, denom, torch.ones_like(denom)),
                        torch.zeros_like(xb))
        c = _e2m1_codes(y.reshape(x.shape[0], k))
        pairs = (c[:, 0::2] | (c[:, 1::2] << 4)).reshape(x.shape[0], k // 32, 4, 4)
        codes[r0:r0 + step] = pairs.transpose(2, 3).reshape(x.shape[0], k // 2)

    list(_POOL.map(blk, range(0, n_rows, step)))
    # scale blocks by 16-row group: [G][K/16][16], rows within a group in the
    # order 0, 8, 1, 9, ..., 7, 15 (rows past N zero)
    groups = -(-n_rows // 16)
    padded = torch.zeros((groups * 16, nb), dtype=torch.uint8)
    padded[:n_rows] = bsc
    order = torch.tensor([r // 2 + 8 * (r % 2) for r in range(16)])
    grouped = padded.view(groups, 16, nb)[:, order, :].permute(0, 2, 1).contiguous()
    return torch.cat([codes.reshape(-1), grouped.reshape(-1)]), s


@dataclass
class Weight:
    """One stored matrix or vector: raw tensor in its storage format (+ FP8 / FP4
    row scales).  FP4 data is the flat byte buffer of quantize_fp4_rows; `dims`
    holds its [N, K]."""

    data: torch.Tensor                  # f32 / bf16 tensor, uint8 codes (fp8), bytes (fp4)
    dtype: str
    scale: Optional[torch.Tensor] = None  # f32 [rows] for fp8 / fp4
    dims: Optional[Tuple[int, int]] = None

    @property
    def shape(self):
        return tuple(self.dims) if self.dims is not None else tuple(self.data.shape)

    def nbytes(self) -> int:
        n = self.data.numel() * self.data.element_size()
        if self.scale is not None:
            n += self.scale.numel() * 4
        return n


@dataclass
class Workload:
    cfg: DraftConfig
    weights: Dict[str, Weight]           # global names and "l{i}.{name}"
    feats: List[torch.Tensor]            # per sequence [T_s, feat_dim], dense dtype
    inject_calls: List[Tuple[int, int, int, int]]  # (seq, first_pos, count, feat_row0)
    id_last: torch.Tensor                # int32 [n_seq]
    n_past: torch.Tensor                 # int32 [n_seq]
    mismatch: torch.Tensor               # int32 [n_seq], 15 = no mismatch
    tail: torch.Tensor                   # int32 [n_seq, 15], random target tokens
    fills: List[int] = field(default_factory=list)
    offsets: List[int] = field(default_factory=list)

    def positions(self, call: Tuple[int, int, int, int]) -> torch.Tensor:
        _, p0, cnt, _ = call
        return torch.arange(p0, p0 + cnt, dtype=torch.int32)

    def call_feats(self, call: Tuple[int, int, int, int]) -> torch.Tensor:
        seq, _, cnt, r0 = call
        return self.feats[seq][r0:r0 + cnt]

    def weight_bytes(self) -> int:
        names = ["lm_head"] + [f"l{i}.{n}" for i in range(self.cfg.n_layer)
                               for n in ("wq", "wk", "wv", "wo", "gate", "up", "down")]
        return sum(self.weights[n].nbytes() for n in names)


LAYER_ORDER = ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm", "ffn_norm",
               "gate", "up", "down")
PROJ = ("wq", "wk", "wv", "wo", "gate", "up", "down")


def _layer_shape(cfg: DraftConfig, name: str) -> Tuple[int, ...]:
    d, qd, kvd, f, hd = cfg.n_embd, cfg.qd, cfg.kvd, cfg.n_ff, cfg.head_dim
    return {
        "attn_norm": (d,), "ffn_norm": (d,), "q_norm": (hd,), "k_norm": (hd,),
        "wq": (qd, d), "wk": (kvd, d), "wv": (kvd, d), "wo": (d, qd),
        "gate": (f, d), "up": (f, d), "down": (d, f),
    }[name]


_CHUNK = 1 << 22
_POOL = _cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 4))


def _mix(*keys: int) -> int:
    """splitmix64 of a key tuple: the seed of one chunk of one drawn tensor."""
    z = 0x9E3779B97F4A7C15
    for k in keys:
        z = (z ^ (k & 0xFFFFFFFFFFFFFFFF)) * 0xBF58476D1CE4E5B9 & 0xFFFFFFFFFFFFFFFF
        z = (z ^ (z >> 27)) * 0x94D049BB133111EB & 0xFFFFFFFFFFFFFFFF
        z ^= z >> 31
    return z & 0x7FFFFFFFFFFFFFFF


def randn(shape, seed: int, index: int, scale: float = 1.0, shift: float = 0.0,
          dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """shift + scale * N(0,1), tensor number `index` of a workload, stored as `dtype`.
    4 Mi-element chunks: chunk c is drawn in f32 by torch's CPU generator seeded
    with mix(seed, index, c), scaled in f32 and rounded once to `dtype`; chunks
    run in parallel threads (the result does not depend on the thread count)."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=dtype)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = torch.Generator().manual_seed(_mix(seed, index, c))
        x = torch.randn(hi - lo, generator=g, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        if shift != 0.0:
            x.add_(shift)
        out[lo:hi] = x.to(dtype)

    list(_POOL.map(fill, range((n + _CHUNK - 1) // _CHUNK)))
    return out.view(shape)


def make_weights(cfg: DraftConfig, g: torch.Generator = None) -> Dict[str, Weight]:
    """Draw every weight; tensor indices follow the fixed order tok_embd, fc,
    hidden_norm, the layers' [attn_norm, wq, wk, wv, wo, q_norm, k_norm, ffn_norm,
    gate, up, down], out_norm, lm_head."""
    w: Dict[str, Weight] = {}
    counter = [0]

    def draw(shape, scale=1.0, shift=0.0, dtype="f32"):
        counter[0] += 1
        return randn(shape, cfg.seed, counter[0], scale, shift, _TORCH[dtype])

    def proj(shape):
        std = float(np.float32(1.0 / np.sqrt(shape[1])))
        if cfg.weight_dtype == "fp8":
            q, s = quantize_fp8_rows(draw(shape, std))
            return Weight(q, "fp8", s)
        if cfg.weight_dtype == "fp4":
            q, s = quantize_fp4_rows(draw(shape, std))
            return Weight(q, "fp4", s, dims=tuple(shape))
        return Weight(draw(shape, std, dtype=cfg.weight_dtype), cfg.weight_dtype)

    def dense_mat(shape, std):
        return Weight(draw(shape, std, dtype=cfg.dense_dtype), cfg.dense_dtype)

    def norm_vec(n):
        return Weight(draw((n,), 0.02, 1.0, dtype=cfg.dense_dtype), cfg.dense_dtype)

    w["tok_embd"] = dense_mat((cfg.n_vocab, cfg.n_embd), 1.0)
    w["fc"] = dense_mat((cfg.n_embd, cfg.feat_dim), 1.0 / np.sqrt(cfg.feat_dim))
    w["hidden_norm"] = norm_vec(cfg.n_embd)
    for i in range(cfg.n_layer):
        for n in LAYER_ORDER:
            shp = _layer_shape(cfg, n)
            w[f"l{i}.{n}"] = norm_vec(shp[0]) if len(shp) == 1 else proj(shp)
    w["out_norm"] = norm_vec(cfg.n_embd)
    w["lm_head"] = proj((cfg.n_vocab, cfg.n_embd))
    return w


def make_workload(cfg: DraftConfig, weights: Optional[Dict[str, Weight]] = None) -> Workload:
    """The full seeded workload of one configuration (seed = cfg.seed)."""
    g = torch.Generator().manual_seed(cfg.seed)
    w = make_weights(cfg)
    if weights is not None:       # caller-provided replacement weights (same draw order kept)
        w = weights
    fills: List[int] = []
    offsets: List[int] = []
    calls: List[Tuple[int, int, int, int]] = []
    if cfg.inject:
        assert cfg.n_seq == 1
        row = 0
        for p0, cnt in cfg.inject:
            calls.append((0, p0, cnt, row))
            row += cnt
        n_rows = [row]
        n_past = [max(p0 + cnt for p0, cnt in cfg.inject)]
    else:
        fl = torch.randint(cfg.fill_lo, cfg.fill_hi + 1, (cfg.n_seq,), generator=g)
        of = torch.randint(0, cfg.offset_hi + 1, (cfg.n_seq,), generator=g)
        fills = [int(x) for x in fl]
        offsets = [int(x) for x in of]
        n_rows, n_past = [], []
        for s in range(cfg.n_seq):
            calls.append((s, offsets[s], fills[s], 0))
            n_rows.append(fills[s])
            n_past.append(offsets[s] + fills[s])
    feats = [randn((n, cfg.feat_dim), cfg.seed, 10_000 + i, dtype=_TORCH[cfg.dense_dtype])
             for i, n in enumerate(n_rows)]
    id_last = torch.randint(0, cfg.n_vocab, (cfg.n_seq,), generator=g, dtype=torch.int64)
    if cfg.mismatch == "geometric":
        # failures before the first success of a Bernoulli(p) sequence, capped at 15
        u = torch.rand((cfg.n_seq,), generator=g, dtype=torch.float64)
        m = torch.floor(torch.log1p(-u) / np.log1p(-cfg.mismatch_p)).clamp_(max=BLOCK - 1)
    else:
        m = torch.randint(0, BLOCK, (cfg.n_seq,), generator=g)
    tail = torch.randint(0, cfg.n_vocab, (cfg.n_seq, BLOCK - 1), generator=g)
    return Workload(cfg=cfg, weights=w, feats=feats, inject_calls=calls,
                    id_last=id_last.to(torch.int32), n_past=torch.tensor(n_past, dtype=torch.int32),
                    mismatch=m.to(torch.int32), tail=tail.to(torch.int32),
                    fills=fills, offsets=offsets)


def make_targets(drafts: np.ndarray, mismatch: np.ndarray, tail: np.ndarray,
                 n_vocab: int) -> np.ndarray:
    """Target tokens that agree with `drafts` before the drawn mismatch index m,
    differ at m (draft + 1 mod vocab) and are random after it.  m = 15 means the
    whole block agrees."""
    drafts = np.asarray(drafts, dtype=np.int64)
    out = np.array(tail, dtype=np.int64, copy=True)
    for s in range(drafts.shape[0]):
        m = int(mismatch[s])
        out[s, :m] = drafts[s, :m]
        if m < BLOCK - 1:
            out[s, m] = (drafts[s, m] + 1) % n_vocab
    return out.astype(np.int32)


def raw_numpy(t: torch.Tensor) -> np.ndarray:
    """Storage bytes of a tensor as numpy: bf16 -> uint16 bit patterns, f32 -> float32,
    fp8 codes -> uint8, ints unchanged."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
