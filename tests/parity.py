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


# The head step alone (dory.rs fn head: logits = (H h) * logit_scale) on the GPU's own final
# hidden rows: H's rows and h have unit norm, so |H_i . h| <= 1, and an f32 dot product over
# bf16 weights (or over the tensor-core path's two bf16 halves of h, which keep about 16
# mantissa bits) errs by far less than 1e-4 of it. A dropped or misindexed logit scale moves
# a logit by |ls_i - ls_j| * |H_i . h|, orders of magnitude more.
HEAD_TOL = 1e-4


def head_err(orc, h_rows, lg_rows) -> float:
    """Largest |GPU logit - (H h_gpu)_i * ls_i| / max|ls| over the given rows."""
    want = (np.asarray(h_rows, np.float64) @ orc.head.T) * orc.logit_scale
    return float(np.max(np.abs(np.asarray(lg_rows, np.float64) - want)) / np.max(np.abs(orc.logit_scale)))


def logit_bound(orc, cfg, h_err_rows) -> float:
    """Bound on |GPU logit - oracle logit| implied by the rows' hidden max-abs errors: with unit
    rows of H, |H_i . dh| <= |dh|_2 <= sqrt(hidden) * max|dh|; plus the head's own HEAD_TOL."""
    ls = float(np.max(np.abs(orc.logit_scale)))
    return ls * (np.sqrt(cfg.hidden) * float(np.max(h_err_rows)) + HEAD_TOL)


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
        self.max_head_err = 0.0
        self.top1 = []

    def close(self):
        self.gpu.close()

    def _note(self, h_gpu, h_orc, lg_gpu=None, lg_orc=None):
        """Record the hidden error of the rows; for a row with logits, assert the head step on
        the GPU's own hidden row (HEAD_TOL) and the logits against the oracle's (the bound the
        row's hidden error implies), and record top-1 agreement."""
        err = float(np.max(np.abs(h_gpu - h_orc)))
        self.max_hidden_err = max(self.max_hidden_err, err)
        if lg_gpu is not None:
            he = head_err(self.orc, h_gpu, lg_gpu)
            self.max_head_err = max(self.max_head_err, he)
            assert he <= HEAD_TOL, f"head step: {he:.3e} of max|logit_scale|"
            le = float(np.max(np.abs(lg_gpu - lg_orc)))
            self.max_logit_err = max(self.max_logit_err, le)
            bound = logit_bound(self.orc, self.cfg, np.abs(h_gpu - h_orc))
            assert le <= bound, f"logits differ by {le:.3e}, above the bound {bound:.3e} of the hidden error"
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
        first = len(ids) - rows  # want last: the chunk's last row; want all: every row
        self._note(h_g, h_o)
        for r in range(rows):
            self._note(h_g[first + r], h_o[first + r], lg_g[r], lg_o[r])
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
