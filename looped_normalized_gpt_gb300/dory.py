"""Python binding of the Dory C ABI (include/dory.h): argument marshalling only.

Every step of the forward runs in libdory.so's CUDA kernels. There is no fallback: if
the library is not built, constructing a handle raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

c_int32_p = ctypes.POINTER(ctypes.c_int32)

OK, EINVAL, ENOMEM, ECUDA, ESTATE, ERANGE, EWAIT = 0, -1, -2, -3, -4, -5, -6
KV_PER_LOOP, KV_LAST_LOOP = 0, 1
KV_F32, KV_Q8_2F = 0, 1
W_F32, W_BF16 = 0, 1
WANT = {"none": 0, "last": 1, "all": 2}


class DoryError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dory error {code}: {msg}")
        self.code = code


class ConfigC(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32), ("ffn", ctypes.c_int32), ("vocab", ctypes.c_int32),
        ("nh", ctypes.c_int32), ("nk", ctypes.c_int32), ("hd", ctypes.c_int32),
        ("window", ctypes.c_int32), ("full_window", ctypes.c_int32), ("max_context", ctypes.c_int32),
        ("n_in", ctypes.c_int32), ("n_rec", ctypes.c_int32), ("n_out", ctypes.c_int32),
        ("layer_pattern", ctypes.c_char_p),
        ("rope_theta_sliding", ctypes.c_double), ("rope_theta_full", ctypes.c_double),
        ("max_loops", ctypes.c_int32), ("kv_mode", ctypes.c_int32), ("kv_quant", ctypes.c_int32),
        ("prompt_loops", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
        ("weight_dtype", ctypes.c_int32),
    ]


class LayerWeightsC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "g", "o", "sq", "sg", "gate", "up", "down",
                                                "mlp_sg", "mlp_su", "alpha")]


class WeightsC(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("head", ctypes.c_void_p), ("logit_scale", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeightsC))]


class StatsC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("weight_bytes_device", "kv_bytes_device", "weight_bytes",
                                                "kv_read_bytes", "kv_write_bytes", "launches", "gemm_launches",
                                                "flops")]


# Every entry point of include/dory.h with its argument types.
SIGNATURES = {
    "dory_create": (ctypes.c_int, [ctypes.POINTER(ConfigC), ctypes.POINTER(WeightsC), ctypes.c_void_p,
                                   ctypes.POINTER(ctypes.c_void_p)]),
    "dory_destroy": (ctypes.c_int, [ctypes.c_void_p]),
    "dory_reset": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "dory_rollback": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]),
    "dory_prefill_chunk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "dory_prefill": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "dory_prefill_batch": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]),
    "dory_decode_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                        ctypes.c_int32]),
    "dory_decode_ragged": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                          ctypes.c_void_p]),
    "dory_decode_conf": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                        c_int32_p, ctypes.POINTER(ctypes.c_float)]),
    "dory_logits": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t]),
    "dory_logits_device": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), c_int32_p]),
    "dory_last_error": (ctypes.c_char_p, []),
    "dory_read_hidden": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]),
    "dory_slot_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, c_int32_p, c_int32_p, c_int32_p]),
    "dory_write_kv_rows": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "dory_set_position": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]),
    "dory_read_kv_f32": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "dory_read_kv_q8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "dory_get_stats": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(StatsC)]),
    "dory_q8_quantize_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 2 + [ctypes.c_int32] * 3 + [ctypes.c_void_p] * 7),
}

_LIB = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libdory.so (built in-tree); raise if it is missing."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built: call looped_normalized_gpt_gb300.build.build() first "
                           "(the Dory forward has no CPU or PyTorch fallback)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _ptr(x):
    """Address of a numpy array (host) or of anything with data_ptr() (a device tensor)."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return ctypes.c_void_p(x.data_ptr())
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"], "arrays must be C-contiguous"
        return ctypes.c_void_p(x.ctypes.data)
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    raise TypeError(f"cannot pass {type(x)}")


class Dory:
    """A handle of the CUDA library: weights resident on the GPU, KV rings of max_seqs sequences."""

    def __init__(self, cfg, weights: dict, stream: int | None = None, lib: ctypes.CDLL | None = None):
        self.lib = lib or load_library()
        self.cfg = cfg
        self._pattern = cfg.pattern.encode()
        c = ConfigC(
            hidden=cfg.hidden, ffn=cfg.ffn, vocab=cfg.vocab, nh=cfg.nh, nk=cfg.nk, hd=cfg.hd, window=cfg.window,
            full_window=cfg.full_window, max_context=cfg.max_context, n_in=cfg.n_in, n_rec=cfg.n_rec,
            n_out=cfg.n_out, layer_pattern=self._pattern, rope_theta_sliding=cfg.rope_theta_sliding,
            rope_theta_full=cfg.rope_theta_full, max_loops=cfg.max_loops,
            kv_mode=KV_PER_LOOP if cfg.kv_mode == "per_loop" else KV_LAST_LOOP,
            kv_quant=KV_Q8_2F if cfg.kv_quant == "q8_2f" else KV_F32, prompt_loops=cfg.prompt_loops,
            max_batch=cfg.max_batch, max_seqs=cfg.max_seqs,
            weight_dtype=W_BF16 if cfg.weight_dtype == "bf16" else W_F32)
        keep = []

        def p(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            keep.append(a)
            return a.ctypes.data

        layers = (LayerWeightsC * len(weights["layers"]))()
        for i, L in enumerate(weights["layers"]):
            if L["kind"] == "attn":
                layers[i] = LayerWeightsC(q=p(L["q"]), k=p(L["k"]), v=p(L["v"]), g=p(L["g"]), o=p(L["o"]),
                                          sq=p(L["sq"]), sg=p(L["sg"]), alpha=p(L["alpha"]))
            else:
                layers[i] = LayerWeightsC(gate=p(L["gate"]), up=p(L["up"]), down=p(L["down"]),
                                          mlp_sg=p(L["sg"]), mlp_su=p(L["su"]), alpha=p(L["alpha"]))
        w = WeightsC(embed=p(weights["embed"]), head=p(weights["head"]), logit_scale=p(weights["logit_scale"]),
                     layers=layers)
        h = ctypes.c_void_p()
        self._check(self.lib.dory_create(ctypes.byref(c), ctypes.byref(w), ctypes.c_void_p(stream or 0),
                                         ctypes.byref(h)))
        self.h = h

    def _check(self, rc: int) -> None:
        if rc != OK:
            raise DoryError(rc, self.lib.dory_last_error().decode())

    def close(self) -> None:
        if getattr(self, "h", None):
            self.lib.dory_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- forward --------------------------------------------------------------------------

    def prefill_chunk(self, seq: int, ids, pos0: int, loops: int, want: str = "last") -> None:
        ids_a = ids if hasattr(ids, "data_ptr") else np.ascontiguousarray(ids, dtype=np.int32)
        n = int(ids_a.numel() if hasattr(ids_a, "numel") else ids_a.size)
        self._check(self.lib.dory_prefill_chunk(self.h, seq, _ptr(ids_a), n, pos0, loops, WANT[want]))

    def prefill(self, seq: int, ids, pos0: int, loops: int, want: str = "last") -> None:
        """A whole prompt (any length) from pos0, as consecutive 64-row chunks."""
        ids_a = ids if hasattr(ids, "data_ptr") else np.ascontiguousarray(ids, dtype=np.int32)
        n = int(ids_a.numel() if hasattr(ids_a, "numel") else ids_a.size)
        self._check(self.lib.dory_prefill(self.h, seq, _ptr(ids_a), n, pos0, loops, WANT[want]))

    def prefill_batch(self, seqs, chunks, loops: int, want: str = "last") -> None:
        """One prefill chunk for each sequence in seqs (chunks[j]: its ids), in one step."""
        seqs_a = np.ascontiguousarray(seqs, dtype=np.int32)
        counts = np.ascontiguousarray([len(c) for c in chunks], dtype=np.int32)
        if len(chunks) and all(hasattr(c, "data_ptr") for c in chunks):
            import torch

            ids_a = torch.cat(list(chunks)).to(torch.int32)
        else:
            ids_a = np.ascontiguousarray(np.concatenate([np.asarray(c) for c in chunks]), dtype=np.int32)
        self._check(self.lib.dory_prefill_batch(self.h, len(seqs_a), _ptr(seqs_a), _ptr(counts), _ptr(ids_a), loops,
                                                WANT[want]))

    def decode_step(self, ids, seqs, loops: int) -> None:
        ids_a = ids if hasattr(ids, "data_ptr") else np.ascontiguousarray(ids, dtype=np.int32)
        seqs_a = np.ascontiguousarray(seqs, dtype=np.int32)
        self._check(self.lib.dory_decode_step(self.h, _ptr(ids_a), _ptr(seqs_a), len(seqs_a), loops))

    def decode_ragged(self, ids, seqs, loops) -> None:
        """One decode token per sequence, each sequence with its own loop count."""
        ids_a = ids if hasattr(ids, "data_ptr") else np.ascontiguousarray(ids, dtype=np.int32)
        seqs_a = np.ascontiguousarray(seqs, dtype=np.int32)
        loops_a = np.ascontiguousarray(loops, dtype=np.int32)
        assert loops_a.size == seqs_a.size, "one loop count per sequence"
        self._check(self.lib.dory_decode_ragged(self.h, _ptr(ids_a), _ptr(seqs_a), len(seqs_a), _ptr(loops_a)))

    def decode_conf(self, token, seq: int, th: float) -> tuple[int, float]:
        """One token under the Conf(th) early-exit gate: (passes, top probability or NaN)."""
        ids_a = token if hasattr(token, "data_ptr") else np.ascontiguousarray([token], dtype=np.int32)
        passes, tp = ctypes.c_int32(), ctypes.c_float()
        self._check(self.lib.dory_decode_conf(self.h, _ptr(ids_a), seq, th, ctypes.byref(passes), ctypes.byref(tp)))
        return passes.value, tp.value

    def logits(self, row: int = 0, out=None) -> np.ndarray:
        dst = out if out is not None else np.empty(self.cfg.vocab, dtype=np.float32)
        cap = dst.numel() if hasattr(dst, "numel") else dst.size
        self._check(self.lib.dory_logits(self.h, row, _ptr(dst), cap))
        return dst

    def logits_device(self) -> tuple[int, int]:
        p = ctypes.c_void_p()
        rows = ctypes.c_int32()
        self._check(self.lib.dory_logits_device(self.h, ctypes.byref(p), ctypes.byref(rows)))
        return p.value, rows.value

    def read_hidden(self, rows: int) -> np.ndarray:
        dst = np.empty((rows, self.cfg.hidden), dtype=np.float32)
        self._check(self.lib.dory_read_hidden(self.h, _ptr(dst), dst.size))
        return dst

    # -- KV state -------------------------------------------------------------------------

    def reset(self, seq: int) -> None:
        self._check(self.lib.dory_reset(self.h, seq))

    def rollback(self, seq: int, n: int) -> None:
        self._check(self.lib.dory_rollback(self.h, seq, n))

    def set_position(self, seq: int, pos: int) -> None:
        self._check(self.lib.dory_set_position(self.h, seq, pos))

    def slot_info(self, ordinal: int) -> tuple[int, int, bool]:
        cap, slots, sl = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        self._check(self.lib.dory_slot_info(self.h, ordinal, ctypes.byref(cap), ctypes.byref(slots),
                                            ctypes.byref(sl)))
        return cap.value, slots.value, bool(sl.value)

    def write_kv_rows(self, seq: int, ordinal: int, slot: int, pos0: int, k, v) -> None:
        k_a = k if hasattr(k, "data_ptr") else np.ascontiguousarray(k, dtype=np.float32)
        v_a = v if hasattr(v, "data_ptr") else np.ascontiguousarray(v, dtype=np.float32)
        n = int(k_a.shape[0])
        self._check(self.lib.dory_write_kv_rows(self.h, seq, ordinal, slot, pos0, n, _ptr(k_a), _ptr(v_a)))

    def read_kv_f32(self, seq: int, ordinal: int, slot: int):
        cap, _, _ = self.slot_info(ordinal)
        nk, hd = self.cfg.nk, self.cfg.hd
        tags = np.empty(cap, np.int32)
        k = np.empty((nk, cap, hd), np.float32)
        v = np.empty((nk, cap, hd), np.float32)
        self._check(self.lib.dory_read_kv_f32(self.h, seq, ordinal, slot, _ptr(tags), _ptr(k), _ptr(v)))
        return tags, k, v

    def read_kv_q8(self, seq: int, ordinal: int, slot: int) -> dict:
        cap, _, _ = self.slot_info(ordinal)
        nk, hd = self.cfg.nk, self.cfg.hd
        out = dict(tags=np.empty(cap, np.int32), kq=np.empty((nk, cap, hd), np.int8),
                   ks=np.empty((nk, cap, hd // 32), np.float32), vq=np.empty((nk, cap, hd), np.int8),
                   vs=np.empty((nk, cap), np.float32), kcol=np.empty((nk, hd), np.float32),
                   vcol=np.empty((nk, hd), np.float32), frozen=np.empty(nk, np.int32))
        self._check(self.lib.dory_read_kv_q8(self.h, seq, ordinal, slot, *[_ptr(out[k]) for k in
                                                                           ("tags", "kq", "ks", "vq", "vs", "kcol",
                                                                            "vcol", "frozen")]))
        return out

    def stats(self) -> dict:
        s = StatsC()
        self._check(self.lib.dory_get_stats(self.h, ctypes.byref(s)))
        return {n: getattr(s, n) for n, _ in StatsC._fields_}
