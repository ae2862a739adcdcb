"""The C-ABI library loads, exports every symbol its header declares, and rejects
bad arguments on the host before touching the GPU (no GPU needed)."""
import ctypes as C

import pytest

from block_diffusion_drafter_fc_gb300.synth import CONFIGS, TEST_CONFIGS, get_config


def _D():
    from block_diffusion_drafter_fc_gb300 import dflash as D
    return D


def test_library_exports_every_header_symbol():
    D = _D()
    syms = D.header_symbols()
    assert len(syms) >= 14
    for s in syms:
        assert hasattr(D.LIB, s), s


def test_struct_layout_matches_header():
    D = _D()
    assert C.sizeof(D.dflash_config) == 80
    assert D.dflash_config.rope_theta.offset == 72
    assert C.sizeof(D.dflash_layer_weights) == 18 * 8
    assert C.sizeof(D.dflash_weights) == 6 * 8 + 16 * 18 * 8


@pytest.mark.parametrize("cfg", list(CONFIGS) + list(TEST_CONFIGS.values()), ids=lambda c: c.name)
def test_workspace_sizes(cfg):
    D = _D()
    rb, sb = D.workspace_size(D.make_config(cfg))
    kv = cfg.n_layer * 2 * cfg.n_head_kv * cfg.window * cfg.head_dim * (2 if cfg.ring_dtype == "bf16" else 4)
    assert rb >= kv * cfg.n_seq + 4 * cfg.n_seq * cfg.window
    assert sb > 0 and sb % 256 == 0


def _bad(**kw):
    D = _D()
    c = D.make_config(get_config("tiny_f32"))
    for k, v in kw.items():
        setattr(c, k, v)
    rb, sb = C.c_size_t(), C.c_size_t()
    return D.LIB.dflash_workspace_size(C.byref(c), C.byref(rb), C.byref(sb))


def test_config_validation():
    assert _bad() == 0
    assert _bad(head_dim=48) == -2          # head_dim must be 32, 64 or 128
    assert _bad(n_head=5, n_head_kv=2) == -2
    assert _bad(n_embd=250) == -2           # K dims multiple of 32
    assert _bad(mask_token_id=512) == -1
    assert _bad(window=0) == -1
    assert _bad(ring_dtype=2) == -2          # FP8 ring not supported
    assert _bad(weight_dtype=7) == -1
    assert _bad(n_layer=17) == -2
    assert _bad(weight_dtype=2, n_embd=288) == -2   # FP8 needs multiples of 64
    assert _bad(weight_dtype=3, n_embd=384) == -2   # FP4 needs multiples of 256
    assert _bad(weight_dtype=4) == -1
    assert _bad(n_head=18, n_head_kv=2, head_dim=128) == -2   # more than 8 q heads per kv head


def test_create_rejects_null_weights_without_gpu():
    D = _D()
    c = D.make_config(get_config("tiny_f32"))
    w = D.dflash_weights()
    h = C.c_void_p()
    assert D.LIB.dflash_create(C.byref(c), C.byref(w), C.c_void_p(256), C.c_void_p(512), C.byref(h)) == -1
    assert D.LIB.dflash_create(None, C.byref(w), None, None, C.byref(h)) == -1
    assert D.LIB.dflash_step(None, 1, None, None, None, None, None) == -1
    assert D.LIB.dflash_status_string(-3).decode().startswith("too many rows")
