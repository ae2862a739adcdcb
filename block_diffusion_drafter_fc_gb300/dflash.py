"""ctypes binding of libdflash (include/dflash.h): argument marshalling only.

Every step of the drafter runs in the library's CUDA kernels.  torch is used
for device memory (the ring, the scratch area, inputs and outputs) and for the
current stream.  Importing this module loads the library; a missing or
unloadable library raises immediately - there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import pathlib
import re
from typing import Dict, List, Optional

import torch

BLOCK = 16          # rows of one noise block (anchor + 15 masks)

PKG = pathlib.Path(__file__).resolve().parent
LIB_PATH = PKG / "libdflash.so"
HEADER = PKG.parent / "include" / "dflash.h"

DTYPE = {"f32": 0, "bf16": 1, "fp8": 2, "fp4": 3}
MAX_LAYERS = 16
PROF_N = 12
PROF_CLASSES = ("embed", "qkv", "attention", "attn_merge", "o_proj", "gate_up", "down", "lm_head",
                "encode", "inject", "accept", "chain")
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported", -3: "too many rows",
          -4: "sequence out of range", -5: "CUDA error", -6: "not captured", -7: "device status"}


class dflash_config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "n_layer", "n_embd", "n_head", "n_head_kv", "head_dim", "n_ff", "window", "n_vocab",
        "n_target_layers", "target_embd", "max_seq", "max_inject", "mask_token_id",
        "weight_dtype", "dense_dtype", "ring_dtype")] + [
        ("eps", C.c_float), ("reserved0", C.c_int32), ("rope_theta", C.c_double)]


_LAYER_PTRS = ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm", "ffn_norm", "gate", "up",
               "down")
_LAYER_SCALES = ("wq_scale", "wk_scale", "wv_scale", "wo_scale", "gate_scale", "up_scale",
                 "down_scale")


class dflash_layer_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _LAYER_PTRS + _LAYER_SCALES]


class dflash_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("tok_embd", "lm_head", "lm_head_scale", "fc",
                                           "hidden_norm", "out_norm")] + [
        ("layers", dflash_layer_weights * MAX_LAYERS)]


class DFlashError(RuntimeError):
    pass


def _load() -> C.CDLL:
    if not LIB_PATH.exists():
        raise DFlashError(f"{LIB_PATH} is missing: build it with block_diffusion_drafter_fc_gb300.build")
    lib = C.CDLL(str(LIB_PATH))
    vp, i32, szp = C.c_void_p, C.c_int32, C.POINTER(C.c_size_t)
    sig = {
        "dflash_workspace_size": (C.c_int, [C.POINTER(dflash_config), szp, szp]),
        "dflash_create": (C.c_int, [C.POINTER(dflash_config), C.POINTER(dflash_weights), vp, vp,
                                    C.POINTER(vp)]),
        "dflash_destroy": (None, [vp]),
        "dflash_encode": (C.c_int, [vp, vp, i32, vp, vp]),
        "dflash_inject": (C.c_int, [vp, i32, vp, vp, i32, vp]),
        "dflash_step": (C.c_int, [vp, i32, vp, vp, vp, vp, vp]),
        "dflash_accept": (C.c_int, [vp, i32, vp, vp, vp, vp]),
        "dflash_capture": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, vp]),
        "dflash_replay": (C.c_int, [vp, vp]),
        "dflash_replay_loop": (C.c_int, [vp, vp]),
        "dflash_graph_nodes": (C.c_int, [vp, i32, C.POINTER(i32), C.POINTER(i32), C.POINTER(i32)]),
        "dflash_profile_stamps": (C.c_int, [vp, i32, C.POINTER(i32), C.POINTER(C.c_double),
                                            C.POINTER(C.c_double), C.POINTER(i32), vp]),
        "dflash_encode_noalloc": (C.c_int, [C.POINTER(dflash_config), vp, vp, vp, i32, vp, vp]),
        "dflash_advance": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, vp]),
        "dflash_set_block_width": (C.c_int, [vp, i32]),
        "dflash_set_chain": (C.c_int, [vp, i32]),
        "dflash_attention_kernel": (C.c_int, [vp, i32]),
        "dflash_capture_loop": (C.c_int, [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
        "dflash_step_host": (C.c_int, [vp, i32, vp, vp, vp, vp, vp]),
        "dflash_ring_reset": (C.c_int, [vp, i32, vp]),
        "dflash_read_status": (C.c_int, [vp, C.POINTER(C.c_uint32), vp]),
        "dflash_profile_enable": (C.c_int, [vp, C.c_int]),
        "dflash_profile_read": (C.c_int, [vp, C.POINTER(C.c_double), C.POINTER(C.c_int32)]),
        "dflash_status_string": (C.c_char_p, [C.c_int]),
        "dflash_last_error": (C.c_char_p, [vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def header_symbols() -> List[str]:
    """Every function the public header declares."""
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^\s*DFLASH_API\s+(?:const\s+)?\w+\s*\*?\s*(dflash_\w+)\s*\(", text, re.M)))


def _check(rc: int, h: Optional[int] = None, what: str = "") -> None:
    if rc != 0:
        msg = LIB.dflash_status_string(rc).decode()
        if h:
            extra = LIB.dflash_last_error(h).decode()
            if extra:
                msg += f" ({extra})"
        raise DFlashError(f"{what}: {msg} [{rc}]")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_config(cfg, max_seq: Optional[int] = None,
                max_inject: Optional[int] = None) -> dflash_config:
    """dflash_config from any object with the drafter's geometry attributes
    (n_layer, n_embd, n_head, n_head_kv, head_dim, n_ff, window, n_vocab,
    n_target_layers, d_t, n_seq, mask_token_id, weight_dtype, dense_dtype,
    ring_dtype as "f32" | "bf16" | "fp8" | "fp4", eps, rope_theta)."""
    c = dflash_config()
    c.n_layer, c.n_embd, c.n_head, c.n_head_kv = cfg.n_layer, cfg.n_embd, cfg.n_head, cfg.n_head_kv
    c.head_dim, c.n_ff, c.window, c.n_vocab = cfg.head_dim, cfg.n_ff, cfg.window, cfg.n_vocab
    c.n_target_layers, c.target_embd = cfg.n_target_layers, cfg.d_t
    c.max_seq = max_seq if max_seq is not None else cfg.n_seq
    c.max_inject = max_inject if max_inject is not None else cfg.window
    c.mask_token_id = cfg.mask_token_id
    c.weight_dtype, c.dense_dtype = DTYPE[cfg.weight_dtype], DTYPE[cfg.dense_dtype]
    c.ring_dtype = DTYPE[cfg.ring_dtype]
    c.eps, c.rope_theta = cfg.eps, cfg.rope_theta
    return c


def workspace_size(c: dflash_config):
    rb, sb = C.c_size_t(), C.c_size_t()
    _check(LIB.dflash_workspace_size(C.byref(c), C.byref(rb), C.byref(sb)), what="workspace_size")
    return rb.value, sb.value


class Drafter:
    """A libdflash handle over the caller's device weights.

    `cfg` is any object with the geometry attributes make_config reads;
    `dev_weights` maps "tok_embd", "lm_head", "fc", "hidden_norm", "out_norm"
    and "l{i}.{attn_norm, wq, wk, wv, wo, q_norm, k_norm, ffn_norm, gate, up,
    down}" to DeviceWeight(data, scale) pairs of device tensors in the stored
    layout the header describes.  The ring and scratch areas are torch uint8
    tensors owned by this object; the weights stay the caller's (kept
    referenced here)."""

    def __init__(self, cfg, dev_weights: Dict[str, "DeviceWeight"],
                 max_seq: Optional[int] = None, max_inject: Optional[int] = None,
                 device: str = "cuda"):
        self.cfg = cfg
        self.c = make_config(cfg, max_seq, max_inject)
        self.ring_bytes, self.scratch_bytes = workspace_size(self.c)
        self.ring_mem = torch.empty(self.ring_bytes + 256, dtype=torch.uint8, device=device)
        self.scratch = torch.empty(self.scratch_bytes + 256, dtype=torch.uint8, device=device)
        self.dev_weights = dev_weights
        w = dflash_weights()
        for n in ("tok_embd", "lm_head", "fc", "hidden_norm", "out_norm"):
            setattr(w, n, dev_weights[n].data.data_ptr())
        if dev_weights["lm_head"].scale is not None:
            w.lm_head_scale = dev_weights["lm_head"].scale.data_ptr()
        for i in range(cfg.n_layer):
            lw = w.layers[i]
            for n in _LAYER_PTRS:
                setattr(lw, n, dev_weights[f"l{i}.{n}"].data.data_ptr())
            for n in ("wq", "wk", "wv", "wo", "gate", "up", "down"):
                sc = dev_weights[f"l{i}.{n}"].scale
                if sc is not None:
                    setattr(lw, n + "_scale", sc.data_ptr())
        self.w = w
        h = C.c_void_p()
        _check(LIB.dflash_create(C.byref(self.c), C.byref(w), self._aligned(self.ring_mem),
                                 self._aligned(self.scratch), C.byref(h)), what="create")
        self.h = h.value

    @staticmethod
    def _aligned(t: torch.Tensor) -> int:
        p = t.data_ptr()
        return (p + 255) // 256 * 256

    def close(self):
        if getattr(self, "h", None):
            LIB.dflash_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- views of caller-visible state
    def ring_views(self):
        """(K, V, ring_pos) as torch views: K/V [max_seq][L][Hkv][W][hd]."""
        cfg, ms = self.cfg, self.c.max_seq
        el = 2 if cfg.ring_dtype == "bf16" else 4
        kv_bytes = cfg.n_layer * 2 * cfg.n_head_kv * cfg.window * cfg.head_dim * el
        base = self._aligned(self.ring_mem) - self.ring_mem.data_ptr()
        raw = self.ring_mem[base:base + kv_bytes * ms]
        dt = torch.bfloat16 if cfg.ring_dtype == "bf16" else torch.float32
        kv = raw.view(dt).view(ms, cfg.n_layer, 2, cfg.n_head_kv, cfg.window, cfg.head_dim)
        pos_off = base + (kv_bytes * ms + 255) // 256 * 256
        pos = self.ring_mem[pos_off:pos_off + 4 * ms * cfg.window].view(torch.int32).view(ms, cfg.window)
        return kv[:, :, 0], kv[:, :, 1], pos

    # ---- C-ABI calls (same names)
    def dflash_encode(self, feats: torch.Tensor, H_t: torch.Tensor, stream=None):
        _check(LIB.dflash_encode(self.h, _ptr(feats), feats.shape[0], _ptr(H_t), _stream(stream)),
               self.h, "encode")

    def dflash_inject(self, seq: int, H_t: torch.Tensor, pos: torch.Tensor, stream=None):
        _check(LIB.dflash_inject(self.h, seq, _ptr(H_t), _ptr(pos), pos.shape[0], _stream(stream)),
               self.h, "inject")

    def dflash_step(self, id_last, n_past, logits, drafts, stream=None):
        _check(LIB.dflash_step(self.h, id_last.shape[0], _ptr(id_last), _ptr(n_past), _ptr(logits),
                               _ptr(drafts), _stream(stream)), self.h, "step")

    def dflash_accept(self, drafts, targets, n_ok, stream=None):
        _check(LIB.dflash_accept(self.h, drafts.shape[0], _ptr(drafts), _ptr(targets), _ptr(n_ok),
                                 _stream(stream)), self.h, "accept")

    def dflash_capture(self, id_last, n_past, logits, drafts, targets=None, n_ok=None, stream=None):
        _check(LIB.dflash_capture(self.h, id_last.shape[0], _ptr(id_last), _ptr(n_past),
                                  _ptr(logits), _ptr(drafts), _ptr(targets), _ptr(n_ok),
                                  _stream(stream)), self.h, "capture")

    def dflash_replay(self, stream=None):
        _check(LIB.dflash_replay(self.h, _stream(stream)), self.h, "replay")

    def dflash_replay_loop(self, stream=None):
        _check(LIB.dflash_replay_loop(self.h, _stream(stream)), self.h, "replay_loop")

    def dflash_graph_nodes(self, loop: bool = False):
        """(kernel nodes, memory alloc/free nodes, other nodes) of the captured graph."""
        k, m, o = C.c_int32(), C.c_int32(), C.c_int32()
        _check(LIB.dflash_graph_nodes(self.h, int(loop), C.byref(k), C.byref(m), C.byref(o)),
               self.h, "graph_nodes")
        return k.value, m.value, o.value

    def dflash_set_chain(self, enable: bool):
        _check(LIB.dflash_set_chain(self.h, int(bool(enable))), self.h, "set_chain")

    def dflash_attention_kernel(self, n_seq: int) -> int:
        """Attention kernel of a step of n_seq sequences: 0 split, 1 clusters, 2 stream-K."""
        rc = LIB.dflash_attention_kernel(self.h, int(n_seq))
        _check(min(rc, 0), self.h, "attention_kernel")
        return rc

    def dflash_set_block_width(self, width: int):
        _check(LIB.dflash_set_block_width(self.h, int(width)), self.h, "set_block_width")

    def dflash_advance(self, drafts, targets, feats, id_last, n_past, n_ok, stream=None):
        _check(LIB.dflash_advance(self.h, drafts.shape[0], _ptr(drafts), _ptr(targets), _ptr(feats),
                                  _ptr(id_last), _ptr(n_past), _ptr(n_ok), _stream(stream)),
               self.h, "advance")

    def dflash_capture_loop(self, targets, feats, id_last, n_past, n_ok, logits, drafts, stream=None):
        _check(LIB.dflash_capture_loop(self.h, targets.shape[0], _ptr(targets), _ptr(feats),
                                       _ptr(id_last), _ptr(n_past), _ptr(n_ok), _ptr(logits),
                                       _ptr(drafts), _stream(stream)), self.h, "capture_loop")

    def dflash_step_host(self, id_last: torch.Tensor, n_past: torch.Tensor, drafts: torch.Tensor,
                         logits: Optional[torch.Tensor] = None, stream=None):
        _check(LIB.dflash_step_host(self.h, id_last.shape[0], _ptr(id_last), _ptr(n_past),
                                    _ptr(logits), _ptr(drafts), _stream(stream)), self.h, "step_host")

    def dflash_ring_reset(self, seq: int, stream=None):
        _check(LIB.dflash_ring_reset(self.h, seq, _stream(stream)), self.h, "ring_reset")

    def dflash_read_status(self, stream=None) -> int:
        v = C.c_uint32()
        rc = LIB.dflash_read_status(self.h, C.byref(v), _stream(stream))
        if rc not in (0, -7):
            _check(rc, self.h, "read_status")
        return v.value

    def dflash_profile_enable(self, enable: bool = True):
        _check(LIB.dflash_profile_enable(self.h, int(enable)), self.h, "profile_enable")

    def dflash_profile_read(self):
        ms = (C.c_double * PROF_N)()
        n = (C.c_int32 * PROF_N)()
        _check(LIB.dflash_profile_read(self.h, ms, n), self.h, "profile_read")
        return {PROF_CLASSES[i]: (ms[i], n[i]) for i in range(PROF_N)}

    def dflash_profile_stamps(self, stream=None, max_launches: int = 128):
        """[(class name, start_us, end_us)] of the last recorded step's launches."""
        cls = (C.c_int32 * max_launches)()
        t0 = (C.c_double * max_launches)()
        t1 = (C.c_double * max_launches)()
        n = C.c_int32()
        _check(LIB.dflash_profile_stamps(self.h, max_launches, cls, t0, t1, C.byref(n),
                                         _stream(stream)), self.h, "profile_stamps")
        return [(PROF_CLASSES[cls[i]], t0[i], t1[i]) for i in range(n.value)]


class DeviceWeight:
    """One weight tensor on the device in its stored layout, and its per-row f32
    scales (FP8 / FP4 projections; None otherwise)."""

    def __init__(self, data: torch.Tensor, scale: Optional[torch.Tensor]):
        self.data, self.scale = data, scale
