"""Plant plausible mistakes in the oracle (on the CPU, by patching its
functions) and check that at least one pin fails for each: a dropped term, a
wrong sign or index, a transposed operand, an off-by-one in the window rule."""
import numpy as np
import pytest

import pins
from oracle import dflash_oracle as O

_orig = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}


def _rms_no_eps(x, w, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) * w


def _rms_sum(x, w, eps):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * w


def _rms_no_weight(x, w, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def _rope_sign(x, pos, inv):
    half = x.shape[-1] // 2
    y = _orig["rope_neox"](x, -np.asarray(pos), inv)
    return y if half else y


def _rope_interleaved(x, pos, inv):
    # GPT-J pairing (2j, 2j+1) instead of NEOX (j, j + hd/2)
    half = x.shape[-1] // 2
    perm = np.concatenate([np.arange(0, 2 * half, 2), np.arange(1, 2 * half, 2)])
    inv_perm = np.argsort(perm)
    return _orig["rope_neox"](x[..., perm], pos, inv)[..., inv_perm]


def _rope_pos_plus_one(x, pos, inv):
    return _orig["rope_neox"](x, np.asarray(pos) + 1, inv)


def _inv_freq_half(theta, hd):
    j = np.arange(hd // 2, dtype=np.float64)
    return np.power(np.float64(theta), -j / hd)


def _attention_gqa_mod(q, kb, vb, kr, vr, valid):
    hq, hkv = q.shape[1], kb.shape[1]
    perm = np.array([h % hkv for h in range(hq)])
    group = hq // hkv
    # feed heads so that the original contiguous grouping yields the modulo grouping
    order = np.argsort(np.array([perm[h] * group + (h // hkv) for h in range(hq)]))
    out = _orig["attention"](q[:, order], kb, vb, kr, vr, valid)
    return out[:, np.argsort(order)]


def _attention_no_scale(q, kb, vb, kr, vr, valid):
    return _orig["attention"](q * np.sqrt(q.shape[-1]), kb, vb, kr, vr, valid)


def _mask_le(ring_pos, n_past, window):
    return _orig["ring_mask"](ring_pos, n_past, window + 1)


def _mask_no_past_check(ring_pos, n_past, window):
    p = np.asarray(ring_pos, dtype=np.int64)[None, :]
    q = n_past + np.arange(16)[:, None]
    return (p >= 0) & (q - p < window)


def _attention_causal(q, kb, vb, kr, vr, valid):
    return _orig["_causal_attention"](q, kb, vb, kr, vr, valid)


def _silu_sign(z):
    return z / (1.0 + np.exp(z))


def _accept_count(drafts, targets):
    return (np.asarray(drafts) == np.asarray(targets)).sum(axis=1).astype(np.int32)


def _bf16_truncate(x):
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _e4m3_bias8(codes):
    return _orig["e4m3_to_f64"](codes) / 2.0


def _decode_no_scale(raw, dtype, scale=None):
    return _orig["decode"](raw, dtype, None if dtype != "fp8" else np.ones_like(scale))


def _inject_kv_v_roped(w, layer, H_t, positions, inv_freq):
    k, v = _orig["inject_kv"](w, layer, H_t, positions, inv_freq)
    return k, O.rope_neox(v, positions, inv_freq)


def _inject_kv_no_knorm(w, layer, H_t, positions, inv_freq):
    cfg = w.cfg
    k = O.linear(H_t, w.get(f"l{layer}.wk")).reshape(H_t.shape[0], cfg.n_head_kv, cfg.head_dim)
    k = O.rope_neox(k, positions, inv_freq)
    _, v = _orig["inject_kv"](w, layer, H_t, positions, inv_freq)
    return k, v


def _encode_no_norm_weight(w, feats):
    cfg = w.cfg
    f = O.decode(feats, cfg.dense_dtype)
    return _rms_no_weight(O.linear(f, w.get("fc")), None, cfg.eps)


def _drafts_rows_0_14(logits):
    l32 = np.asarray(logits).astype(np.float32)
    return np.argmax(l32[..., :-1, :], axis=-1).astype(np.int32)


def _block_tokens_anchor_last(cfg, id_last):
    t = np.full((16,), cfg.mask_token_id, dtype=np.int64)
    t[-1] = id_last
    return t


def _logits_no_norm(w, h):
    return O.linear(h, w.get("lm_head"))


def _silu_on_identity(z):
    return z


def _advance_variant(inject_rows, bonus_shift, past_shift):
    def adv(w, rings, drafts, targets, feats, id_last, n_past):
        targets = np.asarray(targets)
        n_ok = _orig["accept"](drafts, targets[:, :15])
        new_id = np.zeros((len(rings),), dtype=np.int32)
        new_np = np.zeros((len(rings),), dtype=np.int32)
        for s, ring in enumerate(rings):
            m = int(n_ok[s])
            p0 = int(n_past[s])
            rows = inject_rows(m)
            H_t = O.encode(w, np.asarray(feats[s])[:rows])
            O.inject(w, ring, H_t, np.arange(p0, p0 + rows))
            new_id[s] = targets[s, min(15, m + bonus_shift)]
            new_np[s] = p0 + m + 1 + past_shift
        return n_ok, new_id, new_np
    return adv


def _fp4_variant(swap_nibbles, block_len, zero_code_half, transpose=True):
    """The oracle's FP4 decode with one planted mistake."""
    def dec(raw, dtype, scale=None):
        if dtype != "fp4":
            return _orig["decode"](raw, dtype, scale)
        r = np.asarray(raw, dtype=np.uint8).reshape(-1)
        n = len(scale)
        groups = -(-n // 16)
        k = 2 * r.size // (n + 2 * groups)
        codes = r[:n * k // 2].reshape(n, k // 2)
        if transpose:
            codes = codes.reshape(n, k // 32, 4, 4).transpose(0, 1, 3, 2).reshape(n, k // 2)
        sb = r[n * k // 2:].reshape(groups, k // 16, 16)
        p = np.arange(16)
        blocks = np.empty((groups * 16, k // 16), dtype=np.uint8)
        blocks[(np.arange(groups)[:, None] * 16 + p // 2 + 8 * (p % 2)).reshape(-1)] = \
            sb.transpose(0, 2, 1).reshape(groups * 16, k // 16)
        blocks = blocks[:n]
        lo, hi = (codes >> 4, codes & 0xF) if swap_nibbles else (codes & 0xF, codes >> 4)
        v = np.empty((n, k), dtype=np.float64)
        v[:, 0::2] = O.e2m1_to_f64(lo)
        v[:, 1::2] = O.e2m1_to_f64(hi)
        if zero_code_half:      # the subnormal code 1 read as 0
            v[:, 0::2][(lo & 7) == 1] = 0.0
            v[:, 1::2][(hi & 7) == 1] = 0.0
        bs = np.repeat(O.e4m3_to_f64(blocks), block_len, axis=1)
        bs = np.concatenate([bs] * (k // bs.shape[1] + 1), axis=1)[:, :k]
        return v * bs * np.asarray(scale, dtype=np.float64)[:, None]
    return dec


def _fp4_scale_rows_plain(raw, dtype, scale=None):
    """FP4 decode that reads the 16 scale bytes of a block in plain row order."""
    if dtype != "fp4":
        return _orig["decode"](raw, dtype, scale)
    r = np.asarray(raw, dtype=np.uint8).reshape(-1).copy()
    n = len(scale)
    groups = -(-n // 16)
    k = 2 * r.size // (n + 2 * groups)
    sb = r[n * k // 2:].reshape(groups, k // 16, 16)
    # un-permute to plain order, then let the original decode re-permute it
    order = np.array([2 * (i % 8) + i // 8 for i in range(16)])
    r[n * k // 2:] = sb[:, :, order].reshape(-1)
    return _orig["decode"](r, dtype, scale)


def _linear_square_transposed(x, w):
    """y = x W for square weights (the operand orientation lost), x W^T otherwise."""
    return x @ (w if w.shape[0] == w.shape[1] else w.T)


class _SwappedWeights:
    """The model's weights with one norm weight read in place of another."""

    def __init__(self, w, read_as):
        self._w, self._read_as = w, read_as

    def __getattr__(self, name):
        return getattr(self._w, name)

    def get(self, name):
        for suffix, other in self._read_as.items():
            if name.endswith(suffix):
                return self._w.get(name[: -len(suffix)] + other)
        return self._w.get(name)


def _step_hidden_reading(read_as):
    def sh(w, rings, tokens, n_past, causal=False):
        return _orig["step_hidden"](_SwappedWeights(w, read_as), rings, tokens, n_past, causal)
    return sh


def _inject_slot_plus_one(w, ring, H_t, positions):
    cfg = w.cfg
    positions = np.asarray(positions, dtype=np.int64)
    inv_freq = O.inv_freq_table(cfg.rope_theta, cfg.head_dim)
    for layer in range(cfg.n_layer):
        k, v = O.inject_kv(w, layer, H_t, positions, inv_freq)
        ks, vs = O.store(k, cfg.ring_dtype), O.store(v, cfg.ring_dtype)
        for t, p in enumerate(positions):
            slot = (int(p) + 1) % cfg.window
            ring.k[layer, :, slot, :] = ks[t]
            ring.v[layer, :, slot, :] = vs[t]
    for p in positions:
        ring.pos[(int(p) + 1) % cfg.window] = int(p)


def _step_hidden_no_attn_residual(w, rings, tokens, n_past, causal=False):
    """The oracle's layer loop with h = attn wo^T instead of h + attn wo^T."""
    cfg = w.cfg
    n_seq, B = tokens.shape
    inv_freq = O.inv_freq_table(cfg.rope_theta, cfg.head_dim)
    hd, hq, hkv = cfg.head_dim, cfg.n_head, cfg.n_head_kv
    h = w.rows("tok_embd", tokens.reshape(-1)).reshape(n_seq, B, cfg.n_embd)
    pos = np.asarray(n_past, dtype=np.int64)[:, None] + np.arange(B)[None, :]
    for layer in range(cfg.n_layer):
        L = f"l{layer}."
        x = O.rmsnorm(h, w.get(L + "attn_norm"), cfg.eps)
        q = O.linear(x, w.get(L + "wq")).reshape(n_seq, B, hq, hd)
        k = O.linear(x, w.get(L + "wk")).reshape(n_seq, B, hkv, hd)
        v = O.linear(x, w.get(L + "wv")).reshape(n_seq, B, hkv, hd)
        q = O.rope_neox(O.rmsnorm(q, w.get(L + "q_norm"), cfg.eps), pos, inv_freq)
        k = O.rope_neox(O.rmsnorm(k, w.get(L + "k_norm"), cfg.eps), pos, inv_freq)
        att = np.zeros((n_seq, B, hq, hd))
        for s in range(n_seq):
            kr, vr = rings[s].values(layer)
            valid = O.ring_mask(rings[s].pos, int(n_past[s]), cfg.window, B)
            att[s] = O.attention(q[s], k[s], v[s], kr, vr, valid)
        h = O.linear(att.reshape(n_seq, B, hq * hd), w.get(L + "wo"))
        x2 = O.rmsnorm(h, w.get(L + "ffn_norm"), cfg.eps)
        mlp = O.silu(O.linear(x2, w.get(L + "gate"))) * O.linear(x2, w.get(L + "up"))
        h = h + O.linear(mlp, w.get(L + "down"))
    return h


def _drafts_ties_highest(logits):
    l32 = np.asarray(logits).astype(np.float32)[..., 1:, :]
    V = l32.shape[-1]
    return (V - 1 - np.argmax(l32[..., ::-1], axis=-1)).astype(np.int32)


def _drafts_in_f64(logits):
    return np.argmax(np.asarray(logits, dtype=np.float64)[..., 1:, :], axis=-1).astype(np.int32)


MUTANTS = {
    "rmsnorm drops eps": ("rmsnorm", _rms_no_eps),
    "rmsnorm sums instead of mean": ("rmsnorm", _rms_sum),
    "rmsnorm drops weight": ("rmsnorm", _rms_no_weight),
    "rope wrong sign": ("rope_neox", _rope_sign),
    "rope interleaved pairs": ("rope_neox", _rope_interleaved),
    "rope position off by one": ("rope_neox", _rope_pos_plus_one),
    "inv_freq exponent halved": ("inv_freq_table", _inv_freq_half),
    "gqa head modulo": ("attention", _attention_gqa_mod),
    "attention without 1/sqrt(hd)": ("attention", _attention_no_scale),
    "attention causal in block": ("attention", _attention_causal),
    "window off by one": ("ring_mask", _mask_le),
    "future ring slots visible": ("ring_mask", _mask_no_past_check),
    "silu sign": ("silu", _silu_sign),
    "silu dropped": ("silu", _silu_on_identity),
    "accept counts all matches": ("accept", _accept_count),
    "bf16 truncation": ("f64_to_bf16", _bf16_truncate),
    "e4m3 wrong bias": ("e4m3_to_f64", _e4m3_bias8),
    "fp8 scale dropped": ("decode", _decode_no_scale),
    "fp4 nibbles swapped": ("decode", _fp4_variant(True, 16, False)),
    "fp4 block of 32 weights": ("decode", _fp4_variant(False, 32, False)),
    "fp4 code 0.5 read as 0": ("decode", _fp4_variant(False, 16, True)),
    "fp4 bytes read in plain order": ("decode", _fp4_variant(False, 16, False, transpose=False)),
    "fp4 scale rows in plain order": ("decode", _fp4_scale_rows_plain),
    "V roped at injection": ("inject_kv", _inject_kv_v_roped),
    "K not normed at injection": ("inject_kv", _inject_kv_no_knorm),
    "encode drops hidden_norm": ("encode", _encode_no_norm_weight),
    "drafts read rows 0..14": ("greedy_drafts", _drafts_rows_0_14),
    "anchor in the last row": ("block_tokens", _block_tokens_anchor_last),
    "output norm dropped": ("logits_from_hidden", _logits_no_norm),
    "advance injects all 16 block rows": ("advance", _advance_variant(lambda m: 16, 0, 0)),
    "advance bonus from the next row": ("advance", _advance_variant(lambda m: m + 1, 1, 0)),
    "advance n_past grows by n_ok": ("advance", _advance_variant(lambda m: m + 1, 0, -1)),
    "advance drops the anchor row": ("advance", _advance_variant(lambda m: m, 0, 0)),
    "square weights transposed": ("linear", _linear_square_transposed),
    "q normed with the k norm weight": ("step_hidden", _step_hidden_reading({"q_norm": "k_norm"})),
    "ffn norm reads the attention norm": ("step_hidden", _step_hidden_reading({"ffn_norm": "attn_norm"})),
    "gate and up swapped": ("step_hidden", _step_hidden_reading({"gate": "up", "up": "gate"})),
    "ring slot off by one": ("inject", _inject_slot_plus_one),
    "attention residual dropped": ("step_hidden", _step_hidden_no_attn_residual),
    "argmax ties to the highest index": ("greedy_drafts", _drafts_ties_highest),
    "drafts decided on float64 logits": ("greedy_drafts", _drafts_in_f64),
}


def _some_pin_fails():
    for pin in pins.ALL_PINS:
        try:
            pin()
        except Exception:        # noqa: BLE001 - any failure or crash counts
            return pin.__name__
    return None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = _some_pin_fails()
    assert caught is not None, f"no pin catches the mutant: {name}"


def test_unmutated_oracle_passes_every_pin():
    assert _some_pin_fails() is None
