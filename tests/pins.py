"""Pins of the fp64 oracle: checks against what the sources and the mathematics fix.

Each pin is a plain function that raises AssertionError when the oracle
disagrees.  `test_oracle_pins.py` runs them; `test_oracle_mutants.py` plants
plausible mistakes in the oracle and checks that some pin catches each one.
The pins compare the oracle with closed forms, with library routines (torch
float64 rms_norm / scaled_dot_product_attention / silu / dtype casts), with
brute force on tiny inputs, with the verifier example of dflash_engine.py
and with the structural invariants of the dflash-ops model card (section
Correctness): ring wraparound, window masking shown by perturbing
out-of-window slots, non-causal joint denoising, determinism.
"""
from __future__ import annotations

import functools
import json
import math
import pathlib

import numpy as np
import torch
import torch.nn.functional as F

from oracle import dflash_oracle as O
from block_diffusion_drafter_fc_gb300.synth import (
    BLOCK, get_config, make_workload, raw_numpy)
import oracle_bridge as OB

GOLDEN = pathlib.Path(__file__).parent / "golden"


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max |diff| {err:.3e} > {tol:.1e}"


@functools.lru_cache(maxsize=None)
def _tiny():
    return make_workload(get_config("tiny_f32"))


@functools.lru_cache(maxsize=None)
def _ragged():
    return make_workload(get_config("ragged_bf16"))


# ---------------------------------------------------------------- RMSNorm

def pin_rmsnorm_hand():
    """x = [3, 4]: mean(x^2) = 12.5, so y = x / sqrt(12.5) * w (dflash_engine.py,
    class RMSNorm)."""
    y = O.rmsnorm(np.array([3.0, 4.0]), np.array([2.0, 0.5]), 0.0)
    _close(y, [2 * 3 / math.sqrt(12.5), 0.5 * 4 / math.sqrt(12.5)], 1e-15, "rmsnorm [3,4]")


def pin_rmsnorm_eps():
    """eps sits inside the square root: ones(4) with eps = 1 give 1/sqrt(2)."""
    y = O.rmsnorm(np.ones(4), np.ones(4), 1.0)
    _close(y, np.full(4, 1 / math.sqrt(2.0)), 1e-15, "rmsnorm eps")


def pin_rmsnorm_vs_torch():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(5, 37, generator=g, dtype=torch.float64) * 3
    w = 1 + 0.1 * torch.randn(37, generator=g, dtype=torch.float64)
    ref = F.rms_norm(x, (37,), w, eps=1e-6)
    _close(O.rmsnorm(x.numpy(), w.numpy(), 1e-6), ref.numpy(), 1e-13, "rmsnorm vs torch")


# ---------------------------------------------------------------- rope

def pin_inv_freq():
    inv = O.inv_freq_table(1e6, 128)
    assert inv.shape == (64,)
    _close(inv[0], 1.0, 0.0, "inv_freq[0]")
    _close(inv[32], 1e-3, 1e-18, "inv_freq[hd/4] = theta^-1/2")
    _close(inv[1:] / inv[:-1], np.full(63, 1e6 ** (-2 / 128)), 1e-14, "inv_freq ratio")


def pin_rope_hand():
    """head_dim 4, pos 1: inv_freq = [1, theta^-1/2]; element j pairs with j + 2."""
    inv = O.inv_freq_table(1e6, 4)
    a1 = 1e6 ** -0.5
    cases = [([1, 0, 0, 0], [math.cos(1), 0, math.sin(1), 0]),
             ([0, 0, 1, 0], [-math.sin(1), 0, math.cos(1), 0]),
             ([0, 1, 0, 0], [0, math.cos(a1), 0, math.sin(a1)])]
    for x, want in cases:
        _close(O.rope_neox(np.array([x], dtype=np.float64), np.array([1]), inv)[0], want,
               1e-15, f"rope {x}")


def pin_rope_identity_norm_relative():
    g = np.random.default_rng(3)
    inv = O.inv_freq_table(1e6, 64)
    x = g.standard_normal((6, 64))
    _close(O.rope_neox(x, np.zeros(6, dtype=np.int64), inv), x, 0.0, "rope at pos 0")
    pos = np.array([1, 5, 99, 2047, 65535, 70000])
    y = O.rope_neox(x, pos, inv)
    _close(y[:, :32] ** 2 + y[:, 32:] ** 2, x[:, :32] ** 2 + x[:, 32:] ** 2, 1e-12, "pair norms")
    q, k = g.standard_normal(64), g.standard_normal(64)
    for p, s, d in [(100, 37, 11), (5, 5, 4000), (0, 63, 65000)]:
        a = O.rope_neox(q[None], np.array([p]), inv)[0] @ O.rope_neox(k[None], np.array([s]), inv)[0]
        b = O.rope_neox(q[None], np.array([p + d]), inv)[0] @ O.rope_neox(k[None], np.array([s + d]), inv)[0]
        _close(a, b, 1e-9, "rope relative position")


def pin_rope_vs_complex():
    """NEOX rope is multiplication of z_j = x_j + i x_{j+hd/2} by exp(i pos inv_freq_j)."""
    g = torch.Generator().manual_seed(11)
    x = torch.randn(9, 3, 128, generator=g, dtype=torch.float64)
    pos = torch.arange(9, dtype=torch.float64) * 977 + 5
    inv = torch.tensor(O.inv_freq_table(1e6, 128))
    z = torch.complex(x[..., :64], x[..., 64:])
    rot = torch.polar(torch.ones(9, 64, dtype=torch.float64), pos[:, None] * inv[None, :])
    zr = z * rot[:, None, :]
    ref = torch.cat([zr.real, zr.imag], dim=-1)
    _close(O.rope_neox(x.numpy(), pos.numpy().astype(np.int64), inv.numpy()), ref.numpy(),
           1e-12, "rope vs complex rotation")


# ---------------------------------------------------------------- formats

def pin_bf16_round_vs_torch():
    """fp32 -> bf16 nearest-even against torch's cast, including exact ties,
    subnormals and the largest finite values."""
    g = np.random.default_rng(5)
    bits = g.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    ties = (g.integers(0, 2 ** 16, size=4000).astype(np.uint32) << 16) | np.uint32(0x8000)
    edge = np.array([0x00000001, 0x00008000, 0x00018000, 0x007FFFFF, 0x7F7F7FFF,
                     0x7F7F8000, 0x3F808000, 0x3F818000, 0x80008000], dtype=np.uint32)
    allb = np.concatenate([bits, ties, edge])
    f = allb.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16(f.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"bf16 rounding differs at {f[bad[:5]]}"


def pin_bf16_decode_all():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_to_f64(bits)
    ok = np.isnan(want)
    assert np.array_equal(np.isnan(got), ok)
    assert np.array_equal(got[~ok], want[~ok]), "bf16 decode"


def pin_e4m3_decode_all():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want)), "e4m3 NaN codes"
    m = ~np.isnan(want)
    assert np.array_equal(got[m], want[m]), "e4m3 decode"


def pin_e2m1_decode_all():
    """The 16 E2M1 codes decode to the format's values: 0, 0.5, 1, 1.5, 2, 3, 4, 6
    (codes 0..7) and their negatives (codes 8..15, with -0)."""
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = O.e2m1_to_f64(np.arange(16))
    assert np.array_equal(got[:8], want) and np.array_equal(got[8:], [-v for v in want])


def pin_fp4_block_decode_bruteforce():
    """A small FP4 matrix (19 rows: a ragged last row group) decoded element by
    element from its flat buffer: code nibble, block scale and row scale each
    located by the stated byte layout, one weight at a time, against the
    oracle's vectorised decode."""
    g = np.random.default_rng(5)
    n, k = 19, 96
    groups = (n + 15) // 16
    buf = g.integers(0, 256, size=n * k // 2 + groups * 16 * (k // 16), dtype=np.uint8)
    sc_off = n * k // 2
    # keep every block scale finite and positive (E4M3 0x7f / 0xff are NaN)
    buf[sc_off:] &= 0x7e
    srow = g.uniform(0.5, 2.0, size=n)
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    want = np.zeros((n, k))
    for r in range(n):
        for c in range(k):
            # the pair index within the 32-weight group is t + 4j, stored at byte 4t + j
            pair = (c % 32) // 2
            byte = r * (k // 2) + 16 * (c // 32) + 4 * (pair % 4) + pair // 4
            nib = (int(buf[byte]) >> (4 * (c % 2))) & 0xF
            v = table[nib & 7] * (-1.0 if nib & 8 else 1.0)
            # rows 16G + (0, 8, 1, 9, ...): row r sits at position 2 (r % 8) + (r % 16) // 8
            pos = 2 * (r % 8) + (r % 16) // 8
            sbyte = sc_off + ((r // 16) * (k // 16) + c // 16) * 16 + pos
            want[r, c] = srow[r] * float(O.e4m3_to_f64(np.array([buf[sbyte]]))[0]) * v
    got = O.decode(buf, "fp4", srow)
    # the three factors are multiplied in another order: a few ulp of |w| <= 5400
    _close(got, want, 1e-11, "fp4 decode")


def pin_fp8_row_scale():
    """y[n] = s[n] * sum_k q[n,k] x[k] (dflash_head.rs, enum DflashQuantization)."""
    g = torch.Generator().manual_seed(13)
    q = torch.randint(0, 256, (6, 40), generator=g, dtype=torch.uint8)
    q[q == 0x7F] = 0x11
    q[q == 0xFF] = 0x91
    s = torch.rand(6, generator=g) + 0.01
    x = torch.randn(40, generator=g, dtype=torch.float64)
    ref = (q.view(torch.float8_e4m3fn).to(torch.float64) * s.double()[:, None]) @ x
    got = O.linear(x.numpy()[None], O.decode(q.numpy(), "fp8", s.numpy()))[0]
    _close(got, ref.numpy(), 1e-12, "fp8 row scale")


def pin_silu_vs_torch():
    z = np.linspace(-30, 30, 1001)
    _close(O.silu(z), F.silu(torch.from_numpy(z)).numpy(), 1e-14, "silu")


# ---------------------------------------------------------------- attention

def _sdpa_reference(q, k_blk, v_blk, k_ring, v_ring, valid):
    """torch float64 scaled_dot_product_attention with an explicit boolean mask and
    grouped kv heads (enable_gqa repeats each kv head over consecutive q heads)."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                       # [1, Hq, 16, hd]
    keys = np.concatenate([np.transpose(k_ring, (1, 0, 2)), k_blk], axis=0)  # [W+16, Hkv, hd]
    vals = np.concatenate([np.transpose(v_ring, (1, 0, 2)), v_blk], axis=0)
    kt = torch.from_numpy(keys).permute(1, 0, 2)[None]
    vt = torch.from_numpy(vals).permute(1, 0, 2)[None]
    mask = torch.from_numpy(np.concatenate([valid, np.ones((q.shape[0], k_blk.shape[0]), bool)], 1))
    out = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask[None, None], enable_gqa=True)
    return out[0].permute(1, 0, 2).numpy()


def pin_attention_vs_sdpa():
    g = np.random.default_rng(17)
    hq, hkv, hd, W = 6, 2, 8, 12
    q = g.standard_normal((BLOCK, hq, hd))
    kb, vb = g.standard_normal((BLOCK, hkv, hd)), g.standard_normal((BLOCK, hkv, hd))
    kr, vr = g.standard_normal((hkv, W, hd)), g.standard_normal((hkv, W, hd))
    ring_pos = np.array([-1, 3, 30, 31, 12, 40, 41, 27, 28, 29, 39, -1])
    valid = O.ring_mask(ring_pos, 42, W)
    _close(O.attention(q, kb, vb, kr, vr, valid), _sdpa_reference(q, kb, vb, kr, vr, valid),
           1e-12, "attention vs sdpa")


def pin_attention_special_cases():
    g = np.random.default_rng(19)
    hd, W = 8, 5
    q = g.standard_normal((BLOCK, 2, hd))
    kb = np.zeros((BLOCK, 1, hd))
    vb = g.standard_normal((BLOCK, 1, hd))
    kr = np.zeros((1, W, hd))
    vr = g.standard_normal((1, W, hd))
    valid = np.zeros((BLOCK, W), bool)
    valid[:, 2] = True
    # all keys zero -> uniform weights: output = mean of the 17 visible values
    want = (vr[0, 2] + vb[:, 0].sum(axis=0)) / 17.0
    out = O.attention(q, kb, vb, kr, vr, valid)
    _close(out, np.broadcast_to(want, out.shape), 1e-13, "attention, all keys zero")
    # one dominant ring key (score ~50 above the zero block keys) -> its value
    u = g.standard_normal(hd)
    q1 = np.broadcast_to(u, (BLOCK, 1, hd)).copy()
    kr2 = np.zeros((1, W, hd))
    kr2[0, 2] = 50.0 * math.sqrt(hd) * u / (u @ u)
    out = O.attention(q1, kb, vb, kr2, vr, valid)
    _close(out[:, 0], np.broadcast_to(vr[0, 2], (BLOCK, hd)), 1e-12, "attention, one dominant key")


def pin_ring_mask_cases():
    """Window rule 0 <= qpos - kpos < window of the dflash-ops model card, with
    empty slots (-1) and positions at or beyond n_past never visible."""
    W, n_past = 64, 80
    pos = np.array([16, 17, 19, 20, 79, 80, -1, 63])
    v = O.ring_mask(pos, n_past, W)
    assert v.shape == (16, 8)
    # row 0 sits at 80: 80 - 16 = 64 is outside, 80 - 17 = 63 inside
    assert not v[0, 0] and v[0, 1]
    # row 3 sits at 83: 19 outside, 20 inside; row 4 (84): 20 outside
    assert not v[3, 2] and v[3, 3] and not v[4, 3]
    assert v[:, 4].all()                 # 79: newest past position, always visible
    assert not v[:, 5].any()             # 80 = n_past: not a past position
    assert not v[:, 6].any()             # empty slot
    assert v[15, 7]                      # 95 - 63 = 32 < 64
    # brute-force count: slot with kpos is visible to rows i with 80 + i - kpos < 64
    for j, p in enumerate(pos):
        for i in range(16):
            want = (0 <= p < n_past) and (n_past + i - p < W)
            assert bool(v[i, j]) == want, (i, p)


# ---------------------------------------------------------------- acceptance

def pin_accept_example():
    ex = json.loads((GOLDEN / "verify_block_example.json").read_text())
    d = np.array([ex["drafts"]])
    t = np.array([ex["targets"]])
    n_ok = int(O.accept(d, t)[0])
    assert n_ok == ex["expect_n_ok"], n_ok
    assert n_ok + 1 == ex["expect_tau"]
    assert t[0, n_ok] == ex["expect_bonus"]


def pin_greedy_drafts_ties_and_rows():
    """Drafts come from block rows 1..15 only, ties go to the lowest index, and
    the decision is taken on fp32 logits: values that differ in float64 but
    round to the same float32 are a tie (dflash-ops model card, Method: greedy
    drafts at rows 1..15, fp32 arithmetic)."""
    V = 12
    logits = np.zeros((2, 16, V))
    logits[:, 0, 9] = 100.0                       # row 0 is never drafted
    for j in range(1, 16):
        a, b = (j * 5) % V, (j * 5 + 3) % V
        lo, hi = min(a, b), max(a, b)
        logits[0, j, hi] = 2.0 + j                # exact tie: the lower index wins
        logits[0, j, lo] = 2.0 + j
        logits[1, j, hi] = 1.0 + 2.0 ** -40       # larger in float64, equal in float32
        logits[1, j, lo] = 1.0
    d = O.greedy_drafts(logits)
    assert d.shape == (2, 15) and d.dtype == np.int32
    for j in range(1, 16):
        a, b = (j * 5) % V, (j * 5 + 3) % V
        assert d[0, j - 1] == min(a, b), (j, d[0, j - 1])
        assert d[1, j - 1] == min(a, b), (j, d[1, j - 1])


def pin_accept_bruteforce():
    g = np.random.default_rng(23)
    for _ in range(200):
        d = g.integers(0, 50, size=(3, 15))
        m = g.integers(0, 16, size=3)
        t = d.copy()
        for s in range(3):
            if m[s] < 15:
                t[s, m[s]] = d[s, m[s]] + 1
                t[s, m[s] + 1:] = g.integers(0, 50, size=14 - m[s])
        assert np.array_equal(O.accept(d, t), m)


# ---------------------------------------------------------------- encode / inject

def _torch_rope(x, pos, inv):
    z = torch.complex(x[..., : x.shape[-1] // 2], x[..., x.shape[-1] // 2:])
    ang = pos[:, None].double() * inv[None, :]
    while ang.dim() < z.dim():
        ang = ang[:, None, :]
    zr = z * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([zr.real, zr.imag], dim=-1)


# ---------------------------------------------------------------- speculative loop turn

def _advance_case(mismatch, seed=31):
    """tiny_f32 after its prefill: synthetic drafts / targets with the first
    mismatch at `mismatch` (15 = none) and random target features."""
    wl = _tiny()
    cfg = wl.cfg
    w, rings, _ = OB.oracle_prefill(wl)
    g = np.random.default_rng(seed)
    drafts = g.integers(0, cfg.n_vocab, size=(1, 15)).astype(np.int32)
    targets = g.integers(0, cfg.n_vocab, size=(1, 16)).astype(np.int32)
    targets[0, :15] = drafts[0]
    if mismatch < 15:
        targets[0, mismatch] = (drafts[0, mismatch] + 1) % cfg.n_vocab
    fdim = cfg.feat_dim
    feats = O.store(g.standard_normal((1, 16, fdim)), cfg.dense_dtype)
    return w, rings, drafts, targets, feats, wl.id_last.numpy()[:1], wl.n_past.numpy()[:1]


def pin_advance_example():
    """The verifier example of dflash_engine.py (block 8: 3 drafts accepted, then
    a mismatch; tau = 4, the last accepted token is the target's token at index 3)
    carried into the 16-row block: n_ok 3, n_past grows by tau, and the next
    anchor is the target's token at index 3; targets after index 3 do not matter."""
    ex = json.loads((GOLDEN / "verify_block_example.json").read_text())
    w, rings, d, t, f, idl, npast = _advance_case(15)
    k = len(ex["drafts"])
    d[0, :k] = ex["drafts"]
    t[0, :k] = ex["targets"]
    t[0, k:] = (d[0, k:15].tolist() + [0])[:16 - k]
    t[0, 5:] = (t[0, 5:] + 7) % 256      # arbitrary after the mismatch
    n_ok, nid, nnp = O.advance(w, rings, d, t, f, idl, npast)
    assert int(n_ok[0]) == ex["expect_n_ok"]
    assert int(nnp[0]) - int(npast[0]) == ex["expect_tau"]
    assert int(nid[0]) == ex["expect_bonus"]


def pin_advance_injects_verified_rows_only():
    """Only block rows 0..m enter the ring, at positions n_past .. n_past + m: the
    ring's positions become the old ones plus exactly those, and perturbing the
    features of rows m+1..15 changes nothing (they are not verified context)."""
    for m in (0, 4, 15):
        w, rings, d, t, f, idl, npast = _advance_case(m)
        before = rings[0].pos.copy()
        _, nid, nnp = O.advance(w, rings, d, t, f, idl, npast)
        p0 = int(npast[0])
        want = before.copy()
        for p in range(p0, p0 + m + 1):
            want[p % w.cfg.window] = p
        assert np.array_equal(rings[0].pos, want), m
        assert int(nnp[0]) == p0 + m + 1 and int(nid[0]) == int(t[0, m])
        w2, rings2, d2, t2, f2, _, _ = _advance_case(m)
        f2 = f2.copy()
        if m < 15:
            f2[0, m + 1:] = O.store(np.asarray(O.decode(f2[0, m + 1:], w2.cfg.dense_dtype)) * -3.0 + 1.0,
                                    w2.cfg.dense_dtype)
        O.advance(w2, rings2, d2, t2, f2, idl, npast)
        for l in range(w.cfg.n_layer):
            assert np.array_equal(rings[0].k[l], rings2[0].k[l]) and np.array_equal(rings[0].v[l], rings2[0].v[l])


def pin_encode_inject_vs_torch():
    """H_t and one layer's stored K/V against a torch float64 composition of
    library ops (linear, rms_norm) and rope as a complex rotation."""
    wl = _ragged()
    w = OB.oracle_weights(wl)
    cfg = wl.cfg
    call = wl.inject_calls[1]
    feats = raw_numpy(wl.call_feats(call))
    H = O.encode(w, feats)
    ft = torch.from_numpy(O.bf16_to_f64(feats))
    ref = F.rms_norm(F.linear(ft, torch.from_numpy(w.get("fc"))), (cfg.n_embd,),
                     torch.from_numpy(w.get("hidden_norm")), eps=cfg.eps)
    _close(H, ref.numpy(), 1e-12, "encode vs torch")
    ring = O.OracleRing(w.cfg)
    pos = wl.positions(call).numpy()
    O.inject(w, ring, H, pos)
    Ht = torch.from_numpy(H)
    inv = torch.from_numpy(O.inv_freq_table(cfg.rope_theta, cfg.head_dim))
    for layer in range(cfg.n_layer):
        k = F.linear(Ht, torch.from_numpy(w.get(f"l{layer}.wk"))).view(-1, cfg.n_head_kv, cfg.head_dim)
        k = F.rms_norm(k, (cfg.head_dim,), torch.from_numpy(w.get(f"l{layer}.k_norm")), eps=cfg.eps)
        k = _torch_rope(k, torch.from_numpy(pos), inv)
        v = F.linear(Ht, torch.from_numpy(w.get(f"l{layer}.wv"))).view(-1, cfg.n_head_kv, cfg.head_dim)
        slots = pos % cfg.window
        kr, vr = ring.values(layer)
        # ring holds bf16: compare within half a bf16 ulp of the reference
        for t in range(len(pos)):
            kk = k[t].numpy()
            _close(kr[:, slots[t], :], kk, float(np.abs(kk).max()) * 2 ** -8, "ring K")
            vv = v[t].numpy()
            _close(vr[:, slots[t], :], vv, float(np.abs(vv).max()) * 2 ** -8, "ring V")
        assert np.array_equal(ring.pos[slots], pos)


# ---------------------------------------------------------------- whole step

def _torch_step(w, rings, id_last, n_past, B=BLOCK):
    """The block step composed from torch float64 library ops: embedding,
    rms_norm, linear, SDPA with an explicit mask and grouped kv heads, silu."""
    cfg = w.cfg
    n_seq = len(id_last)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    inv = T(O.inv_freq_table(cfg.rope_theta, cfg.head_dim))
    tok = torch.full((n_seq, B), cfg.mask_token_id, dtype=torch.int64)
    tok[:, 0] = torch.as_tensor(np.asarray(id_last, dtype=np.int64))
    h = F.embedding(tok, T(w.get("tok_embd")))
    hd, hq, hkv = cfg.head_dim, cfg.n_head, cfg.n_head_kv
    for layer in range(cfg.n_layer):
        L = f"l{layer}."
        x = F.rms_norm(h, (cfg.n_embd,), T(w.get(L + "attn_norm")), eps=cfg.eps)
        q = F.linear(x, T(w.get(L + "wq"))).view(n_seq, B, hq, hd)
        k = F.linear(x, T(w.get(L + "wk"))).view(n_seq, B, hkv, hd)
        v = F.linear(x, T(w.get(L + "wv"))).view(n_seq, B, hkv, hd)
        q = F.rms_norm(q, (hd,), T(w.get(L + "q_norm")), eps=cfg.eps)
        k = F.rms_norm(k, (hd,), T(w.get(L + "k_norm")), eps=cfg.eps)
        outs = []
        for s in range(n_seq):
            pos = torch.arange(B) + int(n_past[s])
            qs = _torch_rope(q[s], pos, inv)
            ks = _torch_rope(k[s], pos, inv)
            kr, vr = rings[s].values(layer)
            p_ = np.asarray(rings[s].pos, dtype=np.int64)[None, :]
            q_ = int(n_past[s]) + np.arange(B)[:, None]
            valid = (p_ >= 0) & (p_ < int(n_past[s])) & (q_ - p_ < cfg.window)
            outs.append(torch.from_numpy(_sdpa_reference(qs.numpy(), ks.numpy(), v[s].numpy(),
                                                         kr, vr, valid)))
        att = torch.stack(outs).reshape(n_seq, B, hq * hd)
        h = h + F.linear(att, T(w.get(L + "wo")))
        x2 = F.rms_norm(h, (cfg.n_embd,), T(w.get(L + "ffn_norm")), eps=cfg.eps)
        h = h + F.linear(F.silu(F.linear(x2, T(w.get(L + "gate")))) * F.linear(x2, T(w.get(L + "up"))),
                         T(w.get(L + "down")))
    hn = F.rms_norm(h, (cfg.n_embd,), T(w.get("out_norm")), eps=cfg.eps)
    return F.linear(hn, T(w.get("lm_head"))).numpy()


def pin_step_vs_torch():
    wl = _ragged()
    w, rings, _ = OB.oracle_prefill(wl)
    logits, drafts = O.step(w, rings, wl.id_last.numpy(), wl.n_past.numpy())
    ref = _torch_step(w, rings, wl.id_last.numpy(), wl.n_past.numpy())
    _close(logits, ref, 1e-10, "step vs torch composition")
    assert np.array_equal(drafts, np.argmax(ref.astype(np.float32)[:, 1:], axis=-1))


def pin_step_width_vs_torch():
    """Narrow blocks (dflash_head.rs, set_block_g: the anchor plus num_drafts
    mask rows, at least 2): the torch composition over B rows, with the window
    rule written out here rather than taken from the oracle."""
    wl = _ragged()
    w, rings, _ = OB.oracle_prefill(wl)
    for B in (2, 5):
        logits, drafts = O.step(w, rings, wl.id_last.numpy(), wl.n_past.numpy(), width=B)
        assert logits.shape[1] == B and drafts.shape[1] == B - 1
        ref = _torch_step(w, rings, wl.id_last.numpy(), wl.n_past.numpy(), B=B)
        _close(logits, ref, 1e-10, f"width {B} step vs torch composition")
        assert np.array_equal(drafts, np.argmax(ref.astype(np.float32)[:, 1:], axis=-1))


def pin_ring_wraparound():
    """Inject 0..79 into a 64-slot ring in two calls: slots 0..15 end up holding
    64..79, and the step equals the one from a fresh ring holding only 16..79."""
    wl = _tiny()
    w, rings, _ = OB.oracle_prefill(wl)
    pos = rings[0].pos
    assert np.array_equal(pos, np.array([p if p >= 16 else p + 64 for p in range(64)]))
    fresh = O.OracleRing(w.cfg)
    feats = raw_numpy(wl.feats[0][16:80])
    O.inject(w, fresh, O.encode(w, feats), np.arange(16, 80))
    a, _ = O.step(w, rings, [int(wl.id_last[0])], [80])
    b, _ = O.step(w, [fresh], [int(wl.id_last[0])], [80])
    _close(a, b, 1e-9, "wraparound vs fresh ring")


def pin_window_masking():
    """With one layer at n_past 80, window 64: the slot holding 16 is outside every
    row's window, so changing it changes nothing; the slot holding 20 is visible to
    rows 0..3 only (row i sees positions >= 17 + i), and the MLP is row-local."""
    wl = _tiny()
    assert wl.cfg.n_layer == 1
    w, rings, _ = OB.oracle_prefill(wl)
    il = [int(wl.id_last[0])]
    base, _ = O.step(w, rings, il, [80])
    r = rings[0].copy()
    r.k[:, :, 16, :] = (r.k[:, :, 16, :] * -3.0 + 1.0).astype(r.k.dtype)
    r.v[:, :, 16, :] = (r.v[:, :, 16, :] * 5.0 - 2.0).astype(r.v.dtype)
    out, _ = O.step(w, [r], il, [80])
    assert np.array_equal(out, base), "out-of-window slot changed the logits"
    r = rings[0].copy()
    r.v[:, :, 20, :] = (r.v[:, :, 20, :] * 5.0 - 2.0).astype(r.v.dtype)
    r.k[:, :, 20, :] = (r.k[:, :, 20, :] * 2.0).astype(r.k.dtype)
    out, _ = O.step(w, [r], il, [80])
    changed = np.abs(out - base).max(axis=-1)[0] > 1e-9
    assert np.array_equal(changed, np.arange(16) <= 3), changed


def pin_noncausal():
    """Changing the token of block row 15 changes rows 0..14 (joint denoising);
    the causal comparison variant leaves them unchanged."""
    wl = _tiny()
    w, rings, _ = OB.oracle_prefill(wl)
    tok = np.stack([O.block_tokens(w.cfg, int(wl.id_last[0]))])
    tok2 = tok.copy()
    tok2[0, 15] = 7
    a = O.step_hidden(w, rings, tok, [80])
    b = O.step_hidden(w, rings, tok2, [80])
    diff = np.abs(a - b).max(axis=-1)[0]
    assert (diff[:15] > 1e-9).all(), diff
    ca = O.step_hidden(w, rings, tok, [80], causal=True)
    cb = O.step_hidden(w, rings, tok2, [80], causal=True)
    assert np.array_equal(ca[0, :15], cb[0, :15])
    assert not np.array_equal(ca, a)


def pin_determinism():
    wl = _tiny()
    w, rings, _ = OB.oracle_prefill(wl)
    a, da = O.step(w, rings, [int(wl.id_last[0])], [80])
    w2, rings2, _ = OB.oracle_prefill(wl)
    b, db = O.step(w2, rings2, [int(wl.id_last[0])], [80])
    assert np.array_equal(a, b) and np.array_equal(da, db)


def pin_relative_position():
    """Shifting every position (ring and block) by 37 moves every slot (37 is not a
    multiple of the window) and leaves the logits unchanged up to the rounding of
    the stored K/V (fp32 ring here: ~2^-24 relative per element, ~1e-7 on logits)."""
    wl = _tiny()
    w = OB.oracle_weights(wl)
    shift = 37
    calls = [(s, p + shift, c, r) for (s, p, c, r) in wl.inject_calls]
    _, r0, _ = OB.oracle_prefill(wl, w)
    _, r1, _ = OB.oracle_prefill(wl, w, calls)
    assert not np.array_equal(r0[0].pos, r1[0].pos)
    a, _ = O.step(w, r0, [int(wl.id_last[0])], [80])
    b, _ = O.step(w, r1, [int(wl.id_last[0])], [80 + shift])
    _close(a, b, 1e-6, "relative position")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
