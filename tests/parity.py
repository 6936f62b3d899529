"""Helpers that drive the CUDA library (through the C ABI) and the CPU oracle on the same
seeded inputs and compare what they produce."""
from __future__ import annotations

import numpy as np

import synth
from oracle import dory_oracle as O

# Tolerances of the spec gates: hidden states max-abs 1e-4 for the fp32 model,
# 2e-2 for bf16 models; top-1 tokens equal on >= 99% of steps.
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def tol_of(cfg) -> float:
    return TOL_F32 if cfg.weight_dtype == "f32" else TOL_BF16


class Pair:
    """The GPU handle and the oracle for one config and seed."""

    def __init__(self, cfg, seed: int, weights=None):
        from looped_normalized_gpt_gb300 import Dory, build

        build()
        self.cfg = cfg
        self.w = weights if weights is not None else synth.weights(cfg, seed)
        self.gpu = Dory(cfg, self.w)
        self.orc = O.DoryOracle(cfg, self.w)
        self.states = [O.SeqState() for _ in range(cfg.max_seqs)]
        self.max_hidden_err = 0.0
        self.max_logit_err = 0.0
        self.top1 = []

    def close(self):
        self.gpu.close()

    def _note(self, h_gpu, h_orc, lg_gpu=None, lg_orc=None):
        self.max_hidden_err = max(self.max_hidden_err, float(np.max(np.abs(h_gpu - h_orc))))
        if lg_gpu is not None:
            self.max_logit_err = max(self.max_logit_err, float(np.max(np.abs(lg_gpu - lg_orc))))
            self.top1.append(int(np.argmax(lg_gpu)) == int(np.argmax(lg_orc)))

    def prefill(self, seq: int, ids, loops: int, want: str = "last"):
        st = self.states[seq]
        pos0 = st.pos
        self.gpu.prefill_chunk(seq, ids, pos0, loops, want)
        lg_o, h_o = self.orc.forward_chunk(st, ids, pos0, loops, want)
        h_g = self.gpu.read_hidden(len(ids))
        if want == "none":
            self._note(h_g, h_o)
            return h_g, h_o, None, None
        rows = 1 if want == "last" else len(ids)
        lg_g = np.stack([self.gpu.logits(r) for r in range(rows)])
        for r in range(rows):
            self._note(h_g, h_o, lg_g[r], lg_o[r])
        return h_g, h_o, lg_g, lg_o

    def decode(self, seqs, ids, loops: int):
        self.gpu.decode_step(ids, seqs, loops)
        lg_o, h_o = self.orc.decode_step([self.states[s] for s in seqs], ids, loops)
        h_g = self.gpu.read_hidden(len(seqs))
        lg_g = np.stack([self.gpu.logits(b) for b in range(len(seqs))])
        for b in range(len(seqs)):
            self._note(h_g[b], h_o[b], lg_g[b], lg_o[b])
        return h_g, h_o, lg_g, lg_o

    def write_context(self, seq: int, n: int, seed: int, start: int = 0):
        """n synthetic unit-norm K/V rows into every slot of every attention layer of `seq`."""
        c = self.cfg
        for ordn in range(self.orc.attn_layers):
            _, slots, _ = self.gpu.slot_info(ordn)
            for sl in range(slots):
                stream = 1000 * seq + 16 * ordn + sl
                k = synth.kv_rows(seed, 2 * stream, n, c.nk, c.hd, start_row=start)
                v = synth.kv_rows(seed, 2 * stream + 1, n, c.nk, c.hd, start_row=start)
                self.gpu.write_kv_rows(seq, ordn, sl, start, k, v)
                self.orc.write_kv_rows(self.states[seq], ordn, sl, start, k, v)
        self.gpu.set_position(seq, start + n)
        self.states[seq].pos = start + n

    def check_rings(self, seq: int, value_tol: float):
        """Ring tags bit-exact against the ring the oracle's slots imply; rows within tol."""
        c = self.cfg
        for (ordn, sl), slot in self.states[seq].slots.items():
            cap, _, _ = self.gpu.slot_info(ordn)
            want_tags = slot.ring_image(cap)
            if c.kv_quant == "q8_2f":
                got = self.gpu.read_kv_q8(seq, ordn, sl)
                tags = got["tags"]
            else:
                tags, k, v = self.gpu.read_kv_f32(seq, ordn, sl)
            assert np.array_equal(tags.astype(np.int64), want_tags), (ordn, sl)
            if c.kv_quant != "q8_2f":
                for rr in np.nonzero(want_tags >= 0)[0]:
                    p = int(want_tags[rr])
                    assert np.max(np.abs(k[:, rr] - slot.k[p])) <= value_tol, (ordn, sl, p)
                    assert np.max(np.abs(v[:, rr] - slot.v[p])) <= value_tol, (ordn, sl, p)
