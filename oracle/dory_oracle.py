"""CPU oracle of the Dory looped normalized-GPT token forward.

TEST INFRASTRUCTURE ONLY. This module exists to check the CUDA path: only the
tests, the smoke check of the package entry point, and the benchmark's CPU
baseline and reference arm may import or run it. The CUDA library never calls
it and shares no code with it.

It restates, step by step and in the pages' order, what the host forward of
the Rust crate cortiq-engine computes (docs.rs source pages
"cortiq_engine/dory.rs" v0.8.78 and "cortiq_engine/kv_cache.rs" v0.8.78):

  * floating point is float64 throughout, except where the pages fix float32:
    the RoPE table entries (dory.rs, fn stack: f64 angle, sin/cos stored as
    f32), the KV store rows (dory.rs, struct KvSlot: f32 rows), and every step
    of the q8_2f KV store (kv_cache.rs, fn quant_row, fn freeze_cols,
    fn append), which is float32 arithmetic exactly as written there;
  * no blocking, fusion or reordering: one chunk at a time, one row and one KV
    head at a time for attention, library matmuls for the projections.

Readings where the pages are silent:
  * rope_inv_freq's body is not on the pages: inv[j] = theta^(-2j/hd) in f64,
    rounded to f32.
  * per_loop with a loop count that changes between steps leaves holes in the
    higher loop slots; attention at position p reads the positions of
    [p-W+1, p] the slot holds and skips the holes (the window counts
    positions, not rows).
  * the q8_2f store of kv_cache.rs serves as the KV store of every Dory slot
    when q8 is chosen; the freeze runs at the first append that finds >= 64
    stored rows; a last_loop rewrite of a chunk's rows is a truncation of those
    rows followed by their re-append (dory.rs, fn attn_layer), with the same
    freeze check at every append.
  * the oracle does not skip attention weights under 1e-12 in the value sum.

Parity pins for every function here live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np

EPS = 1e-6  # dory.rs, const EPS: justnorm's epsilon
MAX_LOOPS = 16  # dory.rs, const MAX_LOOPS
REWIND = 448  # dory.rs, const REWIND: rows a ring keeps past window and chunk
CHUNK_ROWS = 64  # dory.rs, const HOST_CHUNK
KV_COL_WARMUP = 64  # kv_cache.rs, const KV_COL_WARMUP
KV_K_GROUP = 32  # kv_cache.rs, const KV_K_GROUP

F32 = np.float32


# ----------------------------------------------------------------------------------------
# Elementwise pieces (dory.rs: fn justnorm, fn slerp, fn silu_body, fn gate_body, fn soft_body)
# ----------------------------------------------------------------------------------------


def justnorm(x: np.ndarray) -> np.ndarray:
    """x / sqrt(sum x^2 + eps) over the last axis (dory.rs, fn justnorm)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + EPS)


def residual(x: np.ndarray, out: np.ndarray, alpha: np.ndarray) -> np.ndarray:
    """The nGPT residual (dory.rs, fn slerp): x^ + |alpha| (out^ - x^), renormalised."""
    xh = justnorm(x)
    oh = justnorm(out)
    return justnorm(xh + alpha * (oh - xh))


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def silu_mul(g: np.ndarray, u: np.ndarray, sg: np.ndarray, su: np.ndarray) -> np.ndarray:
    """silu(g*sg) * (u*su) (dory.rs, fn silu_body)."""
    x = g * sg
    return x * sigmoid(x) * (u * su)


def softmax(s: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax of one row of scores (dory.rs, fn soft_body)."""
    e = np.exp(s - np.max(s))
    return e / np.sum(e)


# ----------------------------------------------------------------------------------------
# RoPE (dory.rs: fn stack builds the table, fn attn_layer rotates; reading: inv_freq in f64)
# ----------------------------------------------------------------------------------------


def rope_inv_freq(hd: int, theta: float) -> np.ndarray:
    """inv[j] = theta^(-2j/hd) for j < hd/2, f64 rounded to f32."""
    j = np.arange(hd // 2, dtype=np.float64)
    return (float(F32(theta)) ** (-2.0 * j / hd)).astype(F32)


def rope_table(inv: np.ndarray, pos: int) -> tuple[np.ndarray, np.ndarray]:
    """cos and sin halves for one position: angle pos*inv[j] in f64, stored as f32."""
    ang = float(pos) * inv.astype(np.float64)
    return np.cos(ang).astype(F32), np.sin(ang).astype(F32)


def rotate_half_split(x: np.ndarray, cs: np.ndarray, sn: np.ndarray) -> np.ndarray:
    """Rotate pairs (j, j + hd/2): a' = x cos - y sin, b' = y cos + x sin."""
    half = x.shape[-1] // 2
    a, b = x[..., :half], x[..., half:]
    c, s = cs.astype(np.float64), sn.astype(np.float64)
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# ----------------------------------------------------------------------------------------
# q8_2f row store (kv_cache.rs: fn quant_row, fn freeze_cols, fn append, fn attend)
# ----------------------------------------------------------------------------------------


def round_half_away(v: np.ndarray) -> np.ndarray:
    """Round to nearest, ties away from zero (Rust f32::round), exact in f32."""
    v = np.asarray(v, dtype=F32)
    t = np.trunc(v)
    frac = np.abs(v - t)  # exact: v and t share the exponent range
    return (t + np.sign(v) * (frac >= F32(0.5)).astype(F32)).astype(F32)


def quant_row(x: np.ndarray, col: np.ndarray | None, group: int) -> tuple[np.ndarray, np.ndarray]:
    """One row against the per-channel field (empty field = 1), one scale per `group`
    channels: r = x/col; s = max(absmax/127, 1e-12); q = clamp(round(r/s), -127, 127).
    float32 throughout, as kv_cache.rs writes it. Returns (int8 codes, f32 scales)."""
    x = np.asarray(x, dtype=F32)
    r = x if col is None else (x / col).astype(F32)
    n = r.shape[0]
    codes = np.empty(n, dtype=np.int8)
    scales = []
    for g0 in range(0, n, group):
        g1 = min(n, g0 + group)
        seg = r[g0:g1]
        absmax = F32(np.max(np.abs(seg))) if g1 > g0 else F32(0.0)
        s = max(F32(absmax / F32(127.0)), F32(1e-12))
        s = F32(s)
        q = round_half_away((seg / s).astype(F32))
        codes[g0:g1] = np.clip(q, F32(-127.0), F32(127.0)).astype(np.int8)
        scales.append(s)
    return codes, np.asarray(scales, dtype=F32)


def freeze_field(codes: np.ndarray, scales: np.ndarray, group: int):
    """kv_cache.rs fn freeze_cols for one head and one of K/V: dequantise every stored row
    (x = q*s), col[d] = max(sqrt(sum_p x_pd^2 / n), 1e-6) with the sum taken in f32 in
    row order, then requantise every row against col.

    codes: [n][hd] int8, scales: [n][hd/group] f32. Returns (col, codes', scales')."""
    n, hd = codes.shape
    rows = (codes.astype(F32) * np.repeat(scales, group, axis=1)[:, :hd]).astype(F32)
    col = np.zeros(hd, dtype=F32)
    for p in range(n):  # sequential in p, product rounded before the add
        col = (col + (rows[p] * rows[p]).astype(F32)).astype(F32)
    col = np.maximum(np.sqrt((col / F32(n)).astype(F32)).astype(F32), F32(1e-6)).astype(F32)
    new_codes = np.empty_like(codes)
    new_scales = np.empty_like(scales)
    for p in range(n):
        new_codes[p], new_scales[p] = quant_row(rows[p], col, group)
    return col, new_codes, new_scales


class _Rows:
    """Rows indexed by absolute position, grown on demand (storage only)."""

    def __init__(self, shape, dtype):
        self.shape, self.dtype = shape, dtype
        self.a = np.zeros((0,) + shape, dtype)

    def _fit(self, n):
        if n > len(self.a):
            b = np.zeros((max(n, 2 * len(self.a), 64),) + self.shape, self.dtype)
            b[:len(self.a)] = self.a
            self.a = b

    def __getitem__(self, p):
        return self.a[p]

    def __setitem__(self, p, v):
        self._fit(int(p) + 1)
        self.a[p] = v


class Slot:
    """One KV slot of one sequence: rows by absolute position.

    f32: k, v rows as f32 (dory.rs, struct KvSlot). q8_2f: per (row, kv head) int8 K codes
    with one f32 scale per 32 channels, int8 V codes with one f32 scale per row, and
    per-channel fields kcol/vcol frozen after 64 rows (kv_cache.rs, struct LayerKvCache).
    Rows live in arrays indexed by position; `valid` marks the positions the slot holds."""

    def __init__(self, nk: int, hd: int, quant: bool):
        self.nk, self.hd, self.quant = nk, hd, quant
        ng = hd // KV_K_GROUP
        self.positions: list[int] = []  # stored rows in append order
        self.valid = _Rows((), bool)
        self.k = _Rows((nk, hd), F32)
        self.v = _Rows((nk, hd), F32)
        # q8 state
        self.kq = _Rows((nk, hd), np.int8)
        self.ks = _Rows((nk, ng), F32)
        self.vq = _Rows((nk, hd), np.int8)
        self.vs = _Rows((nk,), F32)
        self.kcol: np.ndarray | None = None  # [nk][hd] f32, None until frozen
        self.vcol: np.ndarray | None = None

    @property
    def stored(self) -> int:
        return len(self.positions)

    def _freeze(self) -> None:
        nk, hd = self.nk, self.hd
        kcol = np.zeros((nk, hd), dtype=F32)
        vcol = np.zeros((nk, hd), dtype=F32)
        P = np.asarray(self.positions)
        for h in range(nk):
            col, kc2, ks2 = freeze_field(self.kq.a[P, h], self.ks.a[P, h], KV_K_GROUP)
            kcol[h] = col
            colv, vc2, vs2 = freeze_field(self.vq.a[P, h], self.vs.a[P, h][:, None], hd)
            vcol[h] = colv
            self.kq.a[P, h] = kc2
            self.ks.a[P, h] = ks2
            self.vq.a[P, h] = vc2
            self.vs.a[P, h] = vs2[:, 0]
        self.kcol, self.vcol = kcol, vcol

    def append(self, pos: int, k: np.ndarray, v: np.ndarray) -> None:
        """Append one row ([nk][hd] each) at a position past every stored one."""
        assert not self.positions or pos > self.positions[-1], "rows arrive in position order"
        k = np.asarray(k, dtype=F32).reshape(self.nk, self.hd)
        v = np.asarray(v, dtype=F32).reshape(self.nk, self.hd)
        if self.quant:
            # kv_cache.rs fn append: the freeze comes first, at >= 64 stored rows
            if self.stored >= KV_COL_WARMUP and self.kcol is None:
                self._freeze()
            ng = self.hd // KV_K_GROUP
            kq = np.empty((self.nk, self.hd), np.int8)
            ks = np.empty((self.nk, ng), F32)
            vq = np.empty((self.nk, self.hd), np.int8)
            vs = np.empty(self.nk, F32)
            for h in range(self.nk):
                kq[h], ks[h] = quant_row(k[h], None if self.kcol is None else self.kcol[h], KV_K_GROUP)
                c, s = quant_row(v[h], None if self.vcol is None else self.vcol[h], self.hd)
                vq[h], vs[h] = c, s[0]
            self.kq[pos], self.ks[pos], self.vq[pos], self.vs[pos] = kq, ks, vq, vs
        else:
            self.k[pos], self.v[pos] = k, v
        self.valid[pos] = True
        self.positions.append(pos)

    def truncate(self, n: int) -> None:
        """Drop the last n stored rows (dory.rs fn attn_layer's overwrite, kv_cache.rs
        fn truncate_last). A frozen field stays frozen."""
        for _ in range(min(n, self.stored)):
            self.valid[self.positions.pop()] = False

    def has(self, pos: int) -> bool:
        return 0 <= pos < len(self.valid.a) and bool(self.valid.a[pos])

    def attend(self, qg: np.ndarray, kh: int, p: int, window: int | None) -> np.ndarray:
        """Attention of the query heads of one KV group at position p.

        qg: [rep][hd] f64 queries that share KV head `kh`.
        Keys: the stored positions of [max(p+1-W, 0), p] (dory.rs fn attn_layer).
        f32: s_j = q.k_j/sqrt(hd), a = softmax(s), y = sum a_j v_j.
        q8: s_j = scale * sum_g ks[j,g] <q*kcol, kq_j>_g ; y = (sum_j a_j vs_j vq_j) * vcol
        (kv_cache.rs fn attend_group_upto)."""
        hd = self.hd
        lo = 0 if window is None else max(p + 1 - window, 0)
        span = np.arange(lo, p + 1)
        keys = span[self.valid.a[lo:p + 1]] if len(self.valid.a) > p else \
            np.array([j for j in span if self.has(j)], dtype=np.int64)
        scale = 1.0 / math.sqrt(hd)
        out = np.zeros_like(qg)
        if self.quant:
            codes = self.kq.a[keys, kh].astype(np.float64).reshape(len(keys), -1, KV_K_GROUP)  # [n][g][32]
            kscale = self.ks.a[keys, kh].astype(np.float64)  # [n][g]
            vcodes = self.vq.a[keys, kh].astype(np.float64)
            vscale = self.vs.a[keys, kh].astype(np.float64)
        else:
            K = self.k.a[keys, kh].astype(np.float64)
            V = self.v.a[keys, kh].astype(np.float64)
        for h in range(qg.shape[0]):
            q = qg[h]
            if self.quant:
                qc = q if self.kcol is None else q * self.kcol[kh].astype(np.float64)
                dots = np.einsum("ngc,gc->ng", codes, qc.reshape(-1, KV_K_GROUP))  # per group
                s = scale * np.sum(kscale * dots, axis=1)
                a = softmax(s)
                y = (a * vscale) @ vcodes
                if self.vcol is not None:
                    y = y * self.vcol[kh].astype(np.float64)
            else:
                a = softmax(K @ q * scale)
                y = a @ V
            out[h] = y
        return out

    def ring_image(self, cap: int):
        """The ring a device keeps of this slot: ring row i holds the latest stored position
        p with p mod cap = i (the position tag), or -1."""
        tags = np.full(cap, -1, dtype=np.int64)
        for p in self.positions:
            if p > tags[p % cap]:
                tags[p % cap] = p
        return tags


# ----------------------------------------------------------------------------------------
# The model (dory.rs: fn attn_layer, fn mlp_layer, fn stack, fn forward_host, fn head)
# ----------------------------------------------------------------------------------------


def top_prob(lg) -> np.float32:
    """dory.rs fn top_prob: the largest softmax probability of a row of logits, counting only
    the entries within 20 of the top. top = the row's max (f32); den = the sum, in vocabulary
    order, of exp(x - top) over the x with x - top > -20, the difference in f32 and the exp
    and sum in f64; the result 1/den rounded to f32."""
    lg = np.asarray(lg, dtype=F32)
    top = F32(np.max(lg))
    den = 0.0
    for x in lg:
        t = F32(x - top)
        if t > F32(-20.0):
            den += math.exp(float(t))
    return F32(1.0 / den)


class ExitRate:
    """dory.rs struct ExitRate: the rate of tokens whose first read-out ended them (f32, from
    1.0) and a token counter (u32). probe(): is this token worth a read-out (rate >= 0.35, or
    one token in eight); note(exited): rate += 0.1 (exited - rate), each step rounded to f32."""

    def __init__(self):
        self.rate = F32(1.0)
        self.tokens = 0

    def probe(self) -> bool:
        self.tokens = (self.tokens + 1) % (1 << 32)
        return bool(self.rate >= F32(0.35) or self.tokens % 8 == 0)

    def note(self, exited: bool) -> None:
        diff = F32(F32(1.0 if exited else 0.0) - self.rate)
        self.rate = F32(self.rate + F32(F32(0.1) * diff))


class SeqState:
    """One sequence: slots[(attention ordinal, loop slot)], the next position, and the
    early-exit gate's rate and counts (dory.rs struct DoryState)."""

    def __init__(self):
        self.slots: dict[tuple[int, int], Slot] = {}
        self.pos = 0
        self.exits = ExitRate()
        self.gate_tokens = 0
        self.gate_one = 0


class DoryOracle:
    def __init__(self, cfg, w: dict, widen=None):
        """cfg: synth.DoryConfig; w: synth.weights(...). `widen` maps stored weights to
        float32 values (bf16 bits are widened exactly)."""
        if widen is None:
            from synth import as_f32 as widen  # input decoding only
        self.cfg = cfg
        c = cfg
        if c.nh % c.nk != 0:
            raise ValueError("nh must be a multiple of nk")
        if c.max_loops > MAX_LOOPS:
            raise ValueError(f"at most {MAX_LOOPS} loops")
        f64 = lambda a: np.asarray(widen(a), dtype=np.float64)  # noqa: E731
        self.embed = f64(w["embed"])
        self.head = f64(w["head"])
        self.logit_scale = np.asarray(w["logit_scale"], dtype=np.float64)
        self.layers = []
        ordinal = 0
        for li, (kind, L) in enumerate(zip(c.pattern, w["layers"])):
            if kind == "-":
                self.layers.append(dict(kind="mlp", gate=f64(L["gate"]), up=f64(L["up"]), down=f64(L["down"]),
                                        sg=L["sg"].astype(np.float64), su=L["su"].astype(np.float64),
                                        alpha=L["alpha"].astype(np.float64)))
            else:
                self.layers.append(dict(kind="attn", sliding=(kind == "S"), ordinal=ordinal,
                                        q=f64(L["q"]), k=f64(L["k"]), v=f64(L["v"]), g=f64(L["g"]), o=f64(L["o"]),
                                        sq=L["sq"].astype(np.float64), sg=L["sg"].astype(np.float64),
                                        alpha=L["alpha"].astype(np.float64)))
                ordinal += 1
        self.attn_layers = ordinal
        self.inv = {True: rope_inv_freq(c.hd, c.rope_theta_sliding), False: rope_inv_freq(c.hd, c.rope_theta_full)}

    # -- helpers ------------------------------------------------------------------------

    def is_rec(self, li: int) -> bool:
        return self.cfg.n_in <= li < self.cfg.n_in + self.cfg.n_rec

    def slot_loop(self, li: int, loop_i: int) -> int:
        """dory.rs fn slot_loop: per_loop keeps one slot per loop for recurrent layers."""
        return loop_i if (self.cfg.kv_mode == "per_loop" and self.is_rec(li)) else 0

    def chunk_loops(self, loops: int, want: str) -> int:
        """dory.rs fn chunk_loops: under last_loop, a chunk whose logits nobody reads
        runs min(loops, prompt_loops) passes."""
        c = self.cfg
        if want == "none" and c.prompt_loops > 0 and c.kv_mode == "last_loop":
            return min(loops, c.prompt_loops)
        return loops

    def slot(self, st: SeqState, ordinal: int, sl: int) -> Slot:
        key = (ordinal, sl)
        if key not in st.slots:
            st.slots[key] = Slot(self.cfg.nk, self.cfg.hd, self.cfg.kv_quant == "q8_2f")
        return st.slots[key]

    def window_of(self, sliding: bool):
        c = self.cfg
        if sliding:
            return c.window
        return c.full_window if c.full_window > 0 else None

    # -- sub-layers ---------------------------------------------------------------------

    def attn_layer(self, L: dict, slot: Slot, h: np.ndarray, pos0: int, overwrite: bool) -> np.ndarray:
        """dory.rs fn attn_layer on rows h[t][hidden] at positions pos0.."""
        c = self.cfg
        t = h.shape[0]
        nh, nk, hd = c.nh, c.nk, c.hd
        rep = nh // nk
        q = h @ L["q"].T
        k = h @ L["k"].T
        v = h @ L["v"].T
        g = h @ L["g"].T
        inv = self.inv[L["sliding"]]
        qr = np.empty((t, nh, hd))
        kr = np.empty((t, nk, hd))
        for r in range(t):
            cs, sn = rope_table(inv, pos0 + r)
            qr[r] = justnorm(rotate_half_split(q[r].reshape(nh, hd), cs, sn)) * L["sq"].reshape(nh, hd)
            kr[r] = justnorm(rotate_half_split(k[r].reshape(nk, hd), cs, sn))
        # the chunk's rows join the slot; each row attends only up to itself
        if overwrite:
            slot.truncate(t)
        for r in range(t):
            slot.append(pos0 + r, kr[r], v[r].reshape(nk, hd))
        window = self.window_of(L["sliding"])
        y = np.empty((t, nh, hd))
        for r in range(t):
            for kh in range(nk):
                y[r, kh * rep:(kh + 1) * rep] = slot.attend(qr[r, kh * rep:(kh + 1) * rep], kh, pos0 + r, window)
        y = y.reshape(t, nh * hd) * sigmoid(g * L["sg"])
        y = justnorm(y)  # over the whole nh*hd row
        return y @ L["o"].T

    def mlp_layer(self, L: dict, h: np.ndarray) -> np.ndarray:
        """dory.rs fn mlp_layer."""
        g = h @ L["gate"].T
        u = h @ L["up"].T
        y = justnorm(silu_mul(g, u, L["sg"], L["su"]))
        return y @ L["down"].T

    def run_layer(self, st: SeqState, li: int, loop_i: int, h: np.ndarray, pos0: int,
                  rewrite_out: bool = False) -> np.ndarray:
        """dory.rs fn stack, closure `run`: the sub-layer, then the residual per row.
        `rewrite_out`: an output layer replaces this chunk's rows (the gate's second read-out)."""
        c = self.cfg
        L = self.layers[li]
        if L["kind"] == "attn":
            sl = self.slot_loop(li, loop_i)
            recurrent = self.is_rec(li)
            overwrite = c.kv_mode == "last_loop" and (recurrent or li >= c.n_in + c.n_rec) and loop_i > 0
            overwrite = overwrite or (rewrite_out and li >= c.n_in + c.n_rec)
            out = self.attn_layer(L, self.slot(st, L["ordinal"], sl), h, pos0, overwrite)
        else:
            out = self.mlp_layer(L, h)
        return residual(h, out, L["alpha"])

    # -- a chunk ------------------------------------------------------------------------

    def head_rows(self, h: np.ndarray) -> np.ndarray:
        """dory.rs fn head: (H h) * logit_scale per row."""
        return (h @ self.head.T) * self.logit_scale

    def forward_chunk(self, st: SeqState, ids, pos0: int, loops: int, want: str = "last", gate=None):
        """One chunk of rows at positions pos0..: embed, input block, `loops` recurrent
        passes with the loop mix, output block, head (dory.rs fn stack, fn forward_host,
        fn head). Returns (logits [rows][vocab] or None, final hidden [t][hidden]).

        gate: None, or th of the Conf(th) early-exit gate, which applies to a chunk of one
        row (dory.rs fn stack's early-exit block): one pass; if the sequence's exit rate
        asks for a read-out, the output block and the head on the pass's state, and
        top_prob >= th ends the token with those logits; otherwise a second pass from the
        state and the input, the output block again (rewriting the rows the read-out
        appended) and the head. The rate notes every read-out. `loops` is not used then.
        Reading: the second read-out replaces the first one's output-layer rows in both KV
        modes (the page's comment states that intent; its per_loop branch would append the
        position a second time)."""
        c = self.cfg
        if loops < 1 or loops > c.max_loops:
            raise ValueError("loops out of range")
        if pos0 != st.pos:
            raise ValueError("chunk does not start at the sequence's position")
        ids = np.asarray(ids, dtype=np.int64)
        t = len(ids)
        h = np.zeros((t, c.hidden))
        for r, i in enumerate(ids):
            if 0 <= i < c.vocab:  # an id past the vocabulary leaves a zero row
                h[r] = self.embed[i]
        L = self.chunk_loops(loops, want)
        early = t == 1 and gate is not None
        for li in range(c.n_in):
            h = self.run_layer(st, li, 0, h, pos0)
        inp = h.copy()
        state = inp.copy()
        for i in range(1 if early else L):
            h = justnorm(state + inp)
            for li in range(c.n_in, c.n_in + c.n_rec):
                h = self.run_layer(st, li, i, h, pos0)
            state = justnorm(h)
        exit_logits = None
        if early:
            stay, readout = False, False
            h = state
            if st.exits.probe():
                readout = True
                for li in range(c.n_in + c.n_rec, c.n_layers):
                    h = self.run_layer(st, li, 0, h, pos0)
                lg = self.head_rows(h)
                stay = bool(top_prob(lg[0]) < F32(gate))
                st.exits.note(not stay)
                if not stay:
                    exit_logits = lg
            else:
                stay = True
            if stay:
                h = justnorm(state + inp)
                for li in range(c.n_in, c.n_in + c.n_rec):
                    h = self.run_layer(st, li, 1, h, pos0)
                h = justnorm(h)
                for li in range(c.n_in + c.n_rec, c.n_layers):
                    h = self.run_layer(st, li, int(readout), h, pos0, rewrite_out=readout)
            st.gate_tokens += 1
            st.gate_one += int(not stay)
        else:
            h = state
            for li in range(c.n_in + c.n_rec, c.n_layers):
                h = self.run_layer(st, li, 0, h, pos0)
        st.pos = pos0 + t
        logits = None
        if exit_logits is not None:
            logits = exit_logits if want != "none" else None
        elif want == "last":
            logits = self.head_rows(h[-1:])
        elif want == "all":
            logits = self.head_rows(h)
        return logits, h

    def prefill(self, st: SeqState, ids, loops: int, chunk: int = CHUNK_ROWS):
        """A prompt in chunks of `chunk` rows: only the last chunk's logits are read."""
        out = None
        n = len(ids)
        for a in range(0, n, chunk):
            b = min(n, a + chunk)
            want = "last" if b == n else "none"
            out = self.forward_chunk(st, ids[a:b], st.pos, loops, want)
        return out

    def decode_step(self, states: list, ids, loops):
        """One token for each sequence (a one-row chunk each, logits read). `loops`: one
        count for every sequence, or one per sequence (each row is its own sequence's
        forward, dory.rs fn forward_host with that sequence's loop count)."""
        per_seq = np.broadcast_to(np.asarray(loops, dtype=np.int64), (len(states),))
        logits, hidden = [], []
        for st, i, L in zip(states, ids, per_seq):
            lg, h = self.forward_chunk(st, [int(i)], st.pos, int(L), "last")
            logits.append(lg[0])
            hidden.append(h[0])
        return np.stack(logits), np.stack(hidden)

    def rollback(self, st: SeqState, n: int) -> None:
        """dory.rs DoryState::rollback: forget the rows from position n on. Every slot keeps
        its stored rows at positions < n (a q8_2f field that froze stays frozen, kv_cache.rs
        fn truncate_last drops rows only); the sequence's position becomes min(pos, n)."""
        for slot in st.slots.values():
            slot.truncate(sum(1 for p in slot.positions if p >= n))
        st.pos = min(st.pos, n)

    def write_kv_rows(self, st: SeqState, ordinal: int, sl: int, pos0: int, k, v) -> None:
        """Append synthetic rows [n][nk][hd] to one slot through the normal append path."""
        s = self.slot(st, ordinal, sl)
        for r in range(len(k)):
            s.append(pos0 + r, k[r], v[r])

    def ring_cap(self, sliding: bool) -> int:
        """Rows of a device ring: window + a 64-row chunk + the rewind slack
        (gpu_metal/dory.rs fn run, sl_cap and the full_window ring)."""
        c = self.cfg
        if sliding:
            return c.window + CHUNK_ROWS + REWIND
        if c.full_window > 0:
            return c.full_window + CHUNK_ROWS + REWIND
        return c.max_context
