"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own formulas: closed forms,
invariants, special cases that reduce to a textbook result, values printed on
the pages (tests/golden/page_constants.json) and a brute-force dense
formulation of the whole forward written separately below. A few tests plant a
mistake in the oracle (on the CPU) and check that a pin catches it.
"""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import dory_oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))
rng = np.random.default_rng(7)


def micro(kv_mode="per_loop", loops=2, window=5, **kw):
    """The pages' unit-test model shape (dory.rs tests, fn tiny): hidden 16, ffn 16, 4 q heads
    over 2 kv heads of 8, vocab 11, pattern S-*-S-*-S-*- with 4 physical layers per block."""
    base = dict(name="micro", hidden=16, ffn=16, vocab=11, nh=4, nk=2, hd=8, window=window,
                pattern="S-*-S-*-S-*-", n_in=4, n_rec=4, n_out=4, loops=loops, max_loops=16,
                kv_mode=kv_mode, kv_quant="f32", weight_dtype="f32", sq=4.0, attn_sg=2.0,
                mlp_suv=1.5 / 4.0, logit_scale=3.0, alpha=(0.2, 0.3), max_context=4096, scale_spread=0.5)
    base.update(kw)
    return synth.DoryConfig(**base)


# ------------------------------------------------------------------------------------------
# constants printed on the pages
# ------------------------------------------------------------------------------------------


def test_constants_match_the_pages():
    assert O.EPS == GOLDEN["EPS"]["value"]
    assert O.MAX_LOOPS == GOLDEN["MAX_LOOPS"]["value"]
    assert O.REWIND == GOLDEN["REWIND"]["value"]
    assert O.CHUNK_ROWS == GOLDEN["HOST_CHUNK"]["value"]
    assert O.KV_COL_WARMUP == GOLDEN["KV_COL_WARMUP"]["value"]
    assert O.KV_K_GROUP == GOLDEN["KV_K_GROUP"]["value"]
    cfg = synth.dory2b()
    o = O.DoryOracle.__new__(O.DoryOracle)
    o.cfg = cfg
    assert o.ring_cap(True) == cfg.window + GOLDEN["ring_extra_rows"]["value"] + GOLDEN["REWIND"]["value"] == 1024
    o.cfg = cfg.replace(full_window=8192)
    assert o.ring_cap(False) == 8704


# ------------------------------------------------------------------------------------------
# justnorm, residual, activations, softmax
# ------------------------------------------------------------------------------------------


def test_justnorm_gives_unit_norm_and_keeps_direction():
    x = rng.normal(size=(50, 37)) * rng.uniform(0.1, 30, size=(50, 1))
    y = O.justnorm(x)
    n = np.linalg.norm(y, axis=1)
    # |x| / sqrt(|x|^2 + eps): within eps / (2|x|^2) of 1
    assert np.all(np.abs(n - 1) <= 1e-6 / (2 * np.min(np.sum(x * x, axis=1))) + 1e-15)
    cos = np.sum(x * y, axis=1) / (np.linalg.norm(x, axis=1) * n)
    assert np.allclose(cos, 1, atol=1e-14)
    assert np.all(O.justnorm(np.zeros(5)) == 0)
    # eps enters under the root: a vector of squared norm 1e-6 comes out with norm 1/sqrt(2)
    v = np.full(4, math.sqrt(1e-6 / 4))
    assert abs(np.linalg.norm(O.justnorm(v)) - 1 / math.sqrt(2)) < 1e-12


def test_residual_endpoints_and_closed_form():
    x = rng.normal(size=64) * 3
    out = rng.normal(size=64) * 0.2
    xh = x / np.linalg.norm(x)
    oh = out / np.linalg.norm(out)
    assert np.allclose(O.residual(x, out, np.zeros(64)), xh, atol=2e-6)
    assert np.allclose(O.residual(x, out, np.ones(64)), oh, atol=2e-6)
    # orthogonal unit vectors: the result is ((1-a) x + a o)/|...|
    e1, e2 = np.eye(64)[0], np.eye(64)[1]
    for a in (0.05, 0.3, 0.7):
        r = O.residual(e1 * 5, e2 * 3, np.full(64, a))
        d = math.hypot(1 - a, a)
        assert abs(r[0] - (1 - a) / d) < 2e-6 and abs(r[1] - a / d) < 2e-6


def test_gate_and_silu_reduce_to_their_scalar_forms():
    assert O.sigmoid(np.zeros(3)).tolist() == [0.5] * 3
    g = (np.arange(21) - 10) * 0.37
    u = 0.1 + np.arange(21) * 0.01
    a, b = np.full(21, 1.3), np.full(21, 0.7)
    got = O.silu_mul(g, u, a, b)
    x = g * 1.3
    want = x / (1 + np.exp(-x)) * (u * 0.7)
    assert np.allclose(got, want, rtol=1e-14, atol=0)
    assert O.silu_mul(np.zeros(4), np.ones(4), np.ones(4), np.ones(4)).tolist() == [0] * 4
    # the gate halves y at g = 0
    y = rng.normal(size=8)
    assert np.allclose(y * O.sigmoid(np.zeros(8) * 3), y / 2)


def test_softmax_sums_to_one_and_ignores_shifts():
    s = rng.normal(size=300) * 20
    p = O.softmax(s)
    assert abs(p.sum() - 1) < 1e-14 and np.all(p >= 0)
    assert np.allclose(O.softmax(s + 1234.5), p, rtol=1e-12)
    assert np.argmax(p) == np.argmax(s)


# ------------------------------------------------------------------------------------------
# RoPE
# ------------------------------------------------------------------------------------------


def test_rope_is_a_complex_rotation_of_half_split_pairs():
    hd = 16
    inv = O.rope_inv_freq(hd, 1e4)
    assert inv[0] == 1.0 and np.all(np.diff(inv) < 0)
    assert abs(inv[-1] - 1e4 ** (-(hd - 2) / hd)) < 1e-7 * inv[-1]
    x = rng.normal(size=hd)
    for pos in (0, 1, 17, 4095):
        cs, sn = O.rope_table(inv, pos)
        got = O.rotate_half_split(x, cs, sn)
        z = (x[: hd // 2] + 1j * x[hd // 2:]) * np.exp(1j * pos * inv.astype(np.float64))
        want = np.concatenate([z.real, z.imag])
        assert np.allclose(got, want, atol=1e-6 * np.abs(x).max())  # f32 table entries
        assert abs(np.linalg.norm(got) - np.linalg.norm(x)) < 1e-6
    cs, sn = O.rope_table(inv, 0)
    assert np.array_equal(O.rotate_half_split(x, cs, sn), x)


def test_rope_scores_depend_only_on_relative_position():
    hd = 32
    inv = O.rope_inv_freq(hd, 1e4)
    q, k = rng.normal(size=hd), rng.normal(size=hd)

    def rot(v, p):
        return O.rotate_half_split(v, *O.rope_table(inv, p))

    for d in (0, 3, 100):
        a = rot(q, 500 + d) @ rot(k, 500)
        b = rot(q, 20 + d) @ rot(k, 20)
        assert abs(a - b) < 1e-5


# ------------------------------------------------------------------------------------------
# attention over a slot
# ------------------------------------------------------------------------------------------


def _filled_slot(rows, nk, hd, quant=False, holes=()):
    s = O.Slot(nk, hd, quant)
    K = rng.normal(size=(rows, nk, hd)).astype(np.float32)
    V = rng.normal(size=(rows, nk, hd)).astype(np.float32)
    for p in range(rows):
        if p not in holes:
            s.append(p, K[p], V[p])
    return s, K.astype(np.float64), V.astype(np.float64)


def _masked_dense(q, K, V, p, lo, keep=None):
    """Whole-row attention with -inf outside [lo, p] (and on holes): the textbook form."""
    n = K.shape[0]
    s = np.full(n, -np.inf)
    for j in range(n):
        if lo <= j <= p and (keep is None or keep[j]):
            s[j] = q @ K[j] / math.sqrt(K.shape[1])
    e = np.exp(s - s.max())
    return (e / e.sum()) @ V


def test_windowed_attend_equals_masked_full_row():
    rows = GOLDEN["windowed_attend_widths"]["rows"]
    s, K, V = _filled_slot(rows, 1, 16)
    q = rng.normal(size=(2, 16))
    p = rows - 1
    for w in GOLDEN["windowed_attend_widths"]["value"]:
        got = s.attend(q, 0, p, w)
        for h in range(2):
            want = _masked_dense(q[h], K[:, 0], V[:, 0], p, max(p + 1 - w, 0))
            assert np.allclose(got[h], want, rtol=1e-12, atol=1e-14), w
    # a window of at least the sequence is full causal attention
    assert np.array_equal(s.attend(q, 0, p, rows), s.attend(q, 0, p, None))
    assert np.array_equal(s.attend(q, 0, p, 10 * rows), s.attend(q, 0, p, None))


def test_window_one_returns_the_current_value():
    s, K, V = _filled_slot(12, 2, 8)
    q = rng.normal(size=(3, 8))
    for kh in range(2):
        y = s.attend(q, kh, 7, 1)
        assert np.array_equal(y, np.tile(V[7, kh], (3, 1)))


def test_equal_keys_average_the_values_and_sharp_queries_pick_one():
    s = O.Slot(1, 8, False)
    k = np.ones((1, 8), np.float32) / math.sqrt(8)
    V = rng.normal(size=(9, 1, 8)).astype(np.float32)
    for p in range(9):
        s.append(p, k, V[p])
    y = s.attend(rng.normal(size=(1, 8)), 0, 8, None)
    assert np.allclose(y[0], V[:, 0].astype(np.float64).mean(axis=0), atol=1e-12)
    s2, K, V2 = _filled_slot(20, 1, 8)
    Kn = K[:, 0] / np.linalg.norm(K[:, 0], axis=1, keepdims=True)
    j = 13
    y = s2.attend(np.array([Kn[j] * 4000.0]), 0, 19, None)  # huge s_q: argmax attention
    assert np.allclose(y[0], V2[j, 0], atol=1e-6)


def test_holes_are_skipped_and_the_window_counts_positions():
    holes = {3, 4, 9}
    s, K, V = _filled_slot(15, 1, 8, holes=holes)
    keep = np.array([p not in holes for p in range(15)])
    q = rng.normal(size=(1, 8))
    for w in (1, 4, 6, 100):
        got = s.attend(q, 0, 14, w)
        want = _masked_dense(q[0], K[:, 0], V[:, 0], 14, max(15 - w, 0), keep)
        assert np.allclose(got[0], want, rtol=1e-12)


def test_ring_image_keeps_the_latest_position_per_row():
    s, _, _ = _filled_slot(30, 1, 4, holes={25})
    tags = s.ring_image(8)
    for i in range(8):
        cands = [p for p in range(30) if p % 8 == i and p != 25]
        assert tags[i] == max(cands)


# ------------------------------------------------------------------------------------------
# q8_2f store
# ------------------------------------------------------------------------------------------


def test_round_half_away_from_zero():
    v = np.array([0.5, -0.5, 1.5, 2.5, -2.5, 0.49999997, -0.49999997, 126.5, 3.2, -3.7], np.float32)
    assert O.round_half_away(v).tolist() == [1, -1, 2, 3, -3, 0, -0, 127, 3, -4]


def test_quant_row_grid_and_error_bound():
    for _ in range(20):
        x = (rng.normal(size=128) * rng.uniform(0.01, 10)).astype(np.float32)
        codes, s = O.quant_row(x, None, 32)
        assert s.shape == (4,)
        for g in range(4):
            seg = slice(32 * g, 32 * g + 32)
            assert np.max(np.abs(codes[seg].astype(int))) == GOLDEN["q8_code_limit"]["value"]
            assert np.all(np.abs(codes[seg] * np.float64(s[g]) - x[seg]) <= s[g] / 2 * (1 + 1e-6))
            # codes are round(x/s) wherever x/s is not within an f32 ulp of a tie
            r = x[seg].astype(np.float64) / s[g]
            far = np.abs(np.abs(r - np.trunc(r)) - 0.5) > 1e-5
            assert np.array_equal(codes[seg][far], (np.sign(r) * np.floor(np.abs(r) + 0.5))[far])
    z = np.zeros(64, np.float32)
    c, s = O.quant_row(z, None, 64)
    assert np.all(c == 0) and s[0] == np.float32(GOLDEN["q8_scale_floor"]["value"])
    # against a field: r = x / col is what gets quantised
    col = rng.uniform(0.5, 2, size=32).astype(np.float32)
    x = rng.normal(size=32).astype(np.float32)
    c1, s1 = O.quant_row(x, col, 32)
    c2, s2 = O.quant_row((x / col).astype(np.float32), None, 32)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_freeze_comes_at_the_65th_append_and_col_is_the_rms():
    nk, hd = 2, 64
    s = O.Slot(nk, hd, True)
    K = rng.normal(size=(70, nk, hd)).astype(np.float32) * np.linspace(0.1, 4, hd).astype(np.float32)
    V = rng.normal(size=(70, nk, hd)).astype(np.float32)
    for p in range(64):
        s.append(p, K[p], V[p])
    assert s.kcol is None
    deq = np.stack([[s.kq[p][h] * np.repeat(s.ks[p][h], 32) for h in range(nk)] for p in range(64)]).astype(np.float64)
    s.append(64, K[64], V[64])
    assert s.kcol is not None
    rms = np.sqrt(np.mean(deq ** 2, axis=0))
    assert np.allclose(s.kcol.astype(np.float64), np.maximum(rms, 1e-6), rtol=1e-5)
    # every stored row was requantised against the field: each group's max |code| is 127
    # (the freeze requantises the dequantised rows, not the original ones)
    for p in range(64):
        for h in range(nk):
            assert np.max(np.abs(s.kq[p][h].reshape(-1, 32).astype(int)), axis=1).tolist() == [127] * 2
            r = deq[p, h] / s.kcol[h].astype(np.float64)
            step = np.repeat(s.ks[p][h], 32).astype(np.float64)
            assert np.all(np.abs(s.kq[p][h] * step - r) <= step * 0.5 * (1 + 1e-5))
    # the freeze does not come again
    kcol = s.kcol.copy()
    for p in range(65, 70):
        s.append(p, K[p], V[p])
    assert np.array_equal(kcol, s.kcol)


def test_freeze_sums_the_squares_in_f32_in_row_order():
    """kv_cache.rs fn freeze_cols sums x^2 over the stored rows in f32, one row after another.
    With one row of 4096 (x^2 = 2^24) and 63 rows of 1: in that order every 2^24 + 1 rounds
    back to 2^24 (the tie goes to the even neighbour), so the sum stays 2^24 and the field is
    sqrt(2^24 / 64) = 512 exactly; in the reverse order the ones first add up to 63 and
    63 + 2^24 rounds to 2^24 + 64, so the field is sqrt(2^18 + 1), whose nearest f32 is
    512 + 2^-10. A sum in f64, or pairwise, or in another order, gives other values."""
    hd = 32
    big = (np.full((1, hd), 64, np.int8), np.full((1, 1), 64.0, np.float32))  # x = 64 * 64 = 4096
    one = (np.full((63, hd), 1, np.int8), np.full((63, 1), 1.0, np.float32))  # x = 1
    for rows, want in (((big, one), 512.0), ((one, big), 512.0 + 2.0 ** -10)):
        codes = np.concatenate([r[0] for r in rows])
        scales = np.concatenate([r[1] for r in rows])
        col, _, _ = O.freeze_field(codes, scales, hd)
        assert col.dtype == np.float32
        assert np.all(col == np.float32(want)), (col[0], want)


def test_q8_attend_matches_f32_within_grid():
    nk, hd, rows = 2, 32, 100
    f = O.Slot(nk, hd, False)
    q8 = O.Slot(nk, hd, True)
    chan = np.where(np.arange(hd) % 2 == 0, 4.0, 0.25)
    for p in range(rows):
        k = (rng.uniform(-0.5, 0.5, size=(nk, hd)) * chan).astype(np.float32)
        v = (rng.uniform(-0.5, 0.5, size=(nk, hd)) * chan).astype(np.float32)
        f.append(p, k, v)
        q8.append(p, k, v)
    q = rng.uniform(-0.5, 0.5, size=(1, hd))
    for g in range(nk):
        of, o8 = f.attend(q, g, rows - 1, None)[0], q8.attend(q, g, rows - 1, None)[0]
        scale = max(np.abs(of).max(), 1e-6)
        assert np.all(np.abs(of - o8) <= scale * GOLDEN["q8_out_rel_tol"]["value"] + GOLDEN["q8_out_abs_tol"]["value"])
    # bytes: 1 per code, 4 per scale (4 K groups + 1 V per head and row), fields once
    q8_bytes = rows * nk * (2 * hd + 4 * (hd // 32) + 4) + 2 * nk * hd * 4
    f32_bytes = rows * nk * 2 * hd * 4
    assert q8_bytes < f32_bytes * GOLDEN["q8_memory_ratio_below"]["value"]


def test_q8_probabilities_match_f32():
    """The softmax over q8 scores stays within 0.02 of the f32 one (prob pin of the pages)."""
    nk, hd, rows = 1, 32, 100
    K = rng.uniform(-0.5, 0.5, size=(rows, nk, hd)).astype(np.float32)
    q8 = O.Slot(nk, hd, True)
    for p in range(rows):
        q8.append(p, K[p], K[p])
    q = rng.uniform(-0.5, 0.5, size=hd)
    pf = O.softmax(K[:, 0].astype(np.float64) @ q / math.sqrt(hd))
    sc = np.array([np.dot(q8.ks[p][0].astype(np.float64), (q * q8.kcol[0] * q8.kq[p][0]).reshape(-1, 32).sum(1)) for p in range(rows)])
    p8 = O.softmax(sc / math.sqrt(hd))
    assert np.max(np.abs(pf - p8)) < GOLDEN["q8_prob_tol"]["value"]


# ------------------------------------------------------------------------------------------
# the whole forward: an independent dense formulation (per_loop: every chunking agrees)
# ------------------------------------------------------------------------------------------


def dense_forward(cfg, w, ids, loops):
    """Whole sequence at once per sub-layer, dense -inf masks, complex-number RoPE,
    norms by np.linalg.norm; written separately from the oracle. per_loop semantics."""
    wf = lambda a: synth.as_f32(a).astype(np.float64)  # noqa: E731
    T = len(ids)
    nh, nk, hd = cfg.nh, cfg.nk, cfg.hd
    E = wf(w["embed"])
    X = np.stack([E[i] if i < cfg.vocab else np.zeros(cfg.hidden) for i in ids])

    def nrm(a):
        return a / np.sqrt(np.linalg.norm(a, axis=-1, keepdims=True) ** 2 + 1e-6)

    def rope(v, theta):  # v [T][H][hd]
        half = hd // 2
        inv = np.power(np.float64(np.float32(theta)), -np.arange(0, hd, 2) / hd).astype(np.float32).astype(np.float64)
        ang = np.arange(T)[:, None] * inv[None, :]
        c = np.cos(ang).astype(np.float32).astype(np.float64)[:, None, :]
        s = np.sin(ang).astype(np.float32).astype(np.float64)[:, None, :]
        z = (v[..., :half] + 1j * v[..., half:]) * (c + 1j * s)
        return np.concatenate([z.real, z.imag], axis=-1)

    def attn(L, X, kind):
        Q = (X @ wf(L["q"]).T).reshape(T, nh, hd)
        K = (X @ wf(L["k"]).T).reshape(T, nk, hd)
        Vv = (X @ wf(L["v"]).T).reshape(T, nk, hd).astype(np.float32).astype(np.float64)
        G = X @ wf(L["g"]).T
        theta = cfg.rope_theta_sliding if kind == "S" else cfg.rope_theta_full
        Q = nrm(rope(Q, theta)) * L["sq"].reshape(nh, hd)
        K = nrm(rope(K, theta)).astype(np.float32).astype(np.float64)
        W = cfg.window if kind == "S" else (cfg.full_window or 10 ** 9)
        i = np.arange(T)[:, None]
        j = np.arange(T)[None, :]
        mask = (j <= i) & (j > i - W)
        Y = np.zeros((T, nh, hd))
        for h in range(nh):
            kh = h // (nh // nk)
            S = Q[:, h] @ K[:, kh].T / math.sqrt(hd)
            S = np.where(mask, S, -np.inf)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            Y[:, h] = P @ Vv[:, kh]
        Y = Y.reshape(T, nh * hd) / (1 + np.exp(-G * L["sg"]))
        return nrm(Y) @ wf(L["o"]).T

    def mlp(L, X):
        g = (X @ wf(L["gate"]).T) * L["sg"]
        u = (X @ wf(L["up"]).T) * L["su"]
        return nrm(g / (1 + np.exp(-g)) * u) @ wf(L["down"]).T

    def layer(li, X):
        L = w["layers"][li]
        out = mlp(L, X) if cfg.pattern[li] == "-" else attn(L, X, cfg.pattern[li])
        a = L["alpha"].astype(np.float64)
        xh, oh = nrm(X), nrm(out)
        return nrm(xh + a * (oh - xh))

    for li in range(cfg.n_in):
        X = layer(li, X)
    inp = X
    state = inp
    for _ in range(loops):
        X = nrm(state + inp)
        for li in range(cfg.n_in, cfg.n_in + cfg.n_rec):
            X = layer(li, X)
        state = nrm(X)
    X = state
    for li in range(cfg.n_in + cfg.n_rec, cfg.n_layers):
        X = layer(li, X)
    logits = X @ wf(w["head"]).T * w["logit_scale"].astype(np.float64)
    return X, logits


def _run(cfg, w, ids, chunk, loops, want="last"):
    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    hs, lg = [], []
    for a in range(0, len(ids), chunk):
        l, h = o.forward_chunk(st, ids[a:a + chunk], a, loops, want)
        hs.append(h)
        lg.append(l)
    return o, st, np.concatenate(hs), lg


@pytest.mark.parametrize("chunk", [1, 4, 64])
def test_oracle_equals_dense_brute_force(chunk):
    cfg = micro()
    w = synth.weights(cfg, 11)
    ids = [(i * 7) % 11 for i in range(23)]
    H, L = dense_forward(cfg, w, ids, 2)
    _, _, h, lg = _run(cfg, w, ids, chunk, 2, "all")
    assert np.allclose(h, H, atol=1e-6)  # f32 KV rows and f32 RoPE entries on both sides
    assert np.allclose(np.concatenate(lg), L, atol=1e-5)
    assert np.allclose(np.linalg.norm(h, axis=1), 1, atol=1e-6)


def test_per_loop_logits_do_not_depend_on_the_chunking():
    cfg = micro()
    w = synth.weights(cfg, 12)
    ids = [(i * 7) % 11 for i in range(23)]
    outs = [_run(cfg, w, ids, c, 2)[3][-1] for c in (1, 4, 64)]
    tol = GOLDEN["chunk_invariance_tol"]["value"]
    assert np.max(np.abs(outs[0] - outs[1])) < tol and np.max(np.abs(outs[0] - outs[2])) < tol


def test_the_last_loop_cache_rewrites_a_position_in_place():
    cfg = micro(kv_mode="last_loop")
    w = synth.weights(cfg, 13)
    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    lg, _ = o.forward_chunk(st, [1, 2, 3, 4, 5, 6, 7, 8], 0, 2, "last")
    n = GOLDEN["last_loop_rows_after_8_tokens"]["value"]
    ords = {k[0] for k in st.slots}
    assert ords == set(range(o.attn_layers))
    assert all(k[1] == 0 for k in st.slots)  # one slot per attention layer
    assert all(s.stored == n for s in st.slots.values())
    assert np.all(np.isfinite(lg))


def test_single_chunk_last_loop_equals_per_loop_last_loop():
    """One chunk: last_loop's final rows are per_loop's rows of the last loop, and the logits
    agree (both read the current loop's keys for every row)."""
    for L in (1, 2, 3):
        cfg_p, cfg_l = micro(kv_mode="per_loop"), micro(kv_mode="last_loop")
        w = synth.weights(cfg_p, 14)
        ids = [3, 1, 4, 1, 5, 9, 2, 6, 5]
        op, sp, hp, lp = _run(cfg_p, w, ids, 64, L)
        ol, sl, hl, ll = _run(cfg_l, w, ids, 64, L)
        assert np.allclose(lp[-1], ll[-1], atol=1e-12)
        for li, kind in enumerate(cfg_p.pattern):
            if kind == "-":
                continue
            ordn = op.layers[li]["ordinal"]
            src = (ordn, L - 1) if op.is_rec(li) else (ordn, 0)
            a, b = sp.slots[src], sl.slots[(ordn, 0)]
            for p in range(len(ids)):
                assert np.array_equal(a.k[p], b.k[p]) and np.array_equal(a.v[p], b.v[p])


def test_one_loop_makes_the_modes_identical_over_many_chunks():
    cfg_p, cfg_l = micro(kv_mode="per_loop"), micro(kv_mode="last_loop")
    w = synth.weights(cfg_p, 15)
    ids = [(i * 5) % 11 for i in range(17)]
    _, _, hp, lp = _run(cfg_p, w, ids, 4, 1)
    _, _, hl, ll = _run(cfg_l, w, ids, 4, 1)
    assert np.array_equal(hp, hl)


def test_last_loop_depends_on_the_chunking_when_loops_exceed_one():
    """Under last_loop, earlier chunks hold their last loop's rows: chunking matters."""
    cfg = micro(kv_mode="last_loop")
    w = synth.weights(cfg, 16)
    ids = [(i * 5) % 11 for i in range(12)]
    a = _run(cfg, w, ids, 1, 2)[3][-1]
    b = _run(cfg, w, ids, 12, 2)[3][-1]
    assert np.max(np.abs(a - b)) > 1e-6


def test_prompt_loops_cut_unread_chunks_only():
    cfg = micro(kv_mode="last_loop", prompt_loops=1)
    w = synth.weights(cfg, 17)
    o = O.DoryOracle(cfg, w)
    assert o.chunk_loops(4, "none") == 1 and o.chunk_loops(4, "last") == 4
    o2 = O.DoryOracle(cfg.replace(prompt_loops=0), w)
    s1, s2 = O.SeqState(), O.SeqState()
    o.forward_chunk(s1, [1, 2, 3], 0, 4, "none")
    o2.forward_chunk(s2, [1, 2, 3], 0, 1, "none")
    for key in s1.slots:
        for p in range(3):
            assert np.array_equal(s1.slots[key].k[p], s2.slots[key].k[p])
    assert O.DoryOracle(cfg.replace(kv_mode="per_loop"), w).chunk_loops(4, "none") == 4


def test_an_id_past_the_vocabulary_embeds_as_zero():
    cfg = micro()
    w = synth.weights(cfg, 18)
    H, L = dense_forward(cfg, w, [3, 99, 5], 2)
    _, _, h, lg = _run(cfg, w, [3, 99, 5], 1, 2, "all")
    assert np.allclose(h, H, atol=1e-6)


def test_full_window_caps_full_layers():
    cfg = micro(full_window=3)
    w = synth.weights(cfg, 19)
    ids = [(i * 3) % 11 for i in range(10)]
    H, _ = dense_forward(cfg, w, ids, 2)
    _, _, h, _ = _run(cfg, w, ids, 4, 2)
    assert np.allclose(h, H, atol=1e-6)
    H2, _ = dense_forward(cfg.replace(full_window=0), w, ids, 2)
    assert np.max(np.abs(H2 - H)) > 1e-6


def test_loops_above_the_maximum_are_refused():
    cfg = micro()
    o = O.DoryOracle(cfg, synth.weights(cfg, 20))
    with pytest.raises(ValueError):
        o.forward_chunk(O.SeqState(), [1], 0, 17, "last")
    with pytest.raises(ValueError):
        O.DoryOracle(cfg.replace(max_loops=17), synth.weights(cfg, 20))


# ------------------------------------------------------------------------------------------
# rollback (dory.rs DoryState::rollback, kv_cache.rs fn truncate_last)
# ------------------------------------------------------------------------------------------


def test_rollback_keeps_the_prefix_a_new_turn_extends():
    """The pages' own test of rollback (dory.rs tests, rollback_keeps_the_prefix_a_new_turn_
    extends): per_loop, 9 tokens, roll back to 5, then tokens 5.. again: the logits are those
    of one run over the whole sequence (per_loop logits do not depend on the chunking)."""
    cfg = micro(window=50)
    w = synth.weights(cfg, 21)
    ids = [(i * 3) % 11 for i in range(12)]
    want = _run(cfg, w, ids, 1, 2)[3][-1]
    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    o.forward_chunk(st, ids[:9], 0, 2, "last")
    o.rollback(st, 5)
    assert st.pos == 5
    lg, _ = o.forward_chunk(st, ids[5:], 5, 2, "last")
    assert np.max(np.abs(lg - want)) < 1e-9


def test_rollback_under_last_loop_equals_the_shorter_chunk():
    """Within a chunk a row sees only rows up to itself, at every loop, so rolling a chunk of
    9 back to 5 leaves exactly what a chunk of 5 leaves, under last_loop too; then a new
    turn gives the same logits."""
    cfg = micro(kv_mode="last_loop", window=6)
    w = synth.weights(cfg, 22)
    ids = [(i * 5 + 2) % 11 for i in range(14)]
    o = O.DoryOracle(cfg, w)
    a, b = O.SeqState(), O.SeqState()
    o.forward_chunk(a, ids[:9], 0, 3, "last")
    o.rollback(a, 5)
    o.forward_chunk(b, ids[:5], 0, 3, "last")
    assert a.slots.keys() == b.slots.keys()
    for key in a.slots:
        assert a.slots[key].positions == b.slots[key].positions == list(range(5))
        for p in range(5):
            assert np.allclose(a.slots[key].k[p], b.slots[key].k[p], atol=1e-12)
            assert np.allclose(a.slots[key].v[p], b.slots[key].v[p], atol=1e-12)
    la, _ = o.forward_chunk(a, ids[5:], 5, 3, "last")
    lb, _ = o.forward_chunk(b, ids[5:], 5, 3, "last")
    assert np.max(np.abs(la - lb)) < 1e-9


def test_rollback_past_the_position_changes_nothing_and_to_zero_is_a_reset():
    cfg = micro()
    w = synth.weights(cfg, 23)
    o = O.DoryOracle(cfg, w)
    st = O.SeqState()
    o.forward_chunk(st, [1, 2, 3, 4], 0, 2, "last")
    before = {k: list(s.positions) for k, s in st.slots.items()}
    o.rollback(st, 9)
    assert st.pos == 4 and {k: list(s.positions) for k, s in st.slots.items()} == before
    o.rollback(st, 0)
    assert st.pos == 0 and all(s.stored == 0 for s in st.slots.values())
    l1, _ = o.forward_chunk(st, [5, 6], 0, 2, "last")
    l2, _ = o.forward_chunk(O.SeqState(), [5, 6], 0, 2, "last")
    assert np.max(np.abs(l1 - l2)) < 1e-12


def test_q8_rollback_keeps_a_frozen_field_and_an_open_one_waits_for_64_kept_rows():
    """kv_cache.rs fn truncate_last drops rows and keeps the fields: after the freeze a
    rollback leaves kcol/vcol as they were; before it, only the rows kept count toward the 64
    the freeze waits for, so 50 rows rolled back to 20 and then 45 more rows store exactly
    what 20 + 45 rows store (the freeze at the 65th row reads the same 64 rows)."""
    nk, hd = 2, 64
    r = synth.kv_rows(5, 0, 120, nk, hd) * np.float32(2.0)
    s_ = synth.kv_rows(5, 1, 120, nk, hd) * np.linspace(0.3, 3, hd).astype(np.float32)
    frozen = O.Slot(nk, hd, True)
    for p in range(70):
        frozen.append(p, r[p], s_[p])
    kcol, vcol = frozen.kcol.copy(), frozen.vcol.copy()
    st = O.SeqState()
    st.slots[(0, 0)] = frozen
    st.pos = 70
    O.DoryOracle.rollback(None, st, 30)
    assert frozen.stored == 30 and np.array_equal(frozen.kcol, kcol) and np.array_equal(frozen.vcol, vcol)
    a, b = O.Slot(nk, hd, True), O.Slot(nk, hd, True)
    for p in range(50):
        a.append(p, r[p], s_[p])
    sa = O.SeqState()
    sa.slots[(0, 0)] = a
    sa.pos = 50
    O.DoryOracle.rollback(None, sa, 20)
    assert a.stored == 20 and a.kcol is None
    for p in range(20):
        b.append(p, r[p], s_[p])
    for p in range(20, 65):
        a.append(p, r[100 - p], s_[100 - p])
        b.append(p, r[100 - p], s_[100 - p])
    assert a.kcol is not None and np.array_equal(a.kcol, b.kcol) and np.array_equal(a.vcol, b.vcol)
    for p in range(65):
        assert np.array_equal(a.kq[p], b.kq[p]) and np.array_equal(a.ks[p], b.ks[p])
        assert np.array_equal(a.vq[p], b.vq[p]) and np.array_equal(a.vs[p], b.vs[p])


# ------------------------------------------------------------------------------------------
# the Conf(th) early-exit gate (dory.rs fn stack's early-exit block, fn top_prob, ExitRate)
# ------------------------------------------------------------------------------------------


def test_top_prob_of_a_sure_row_and_of_ties():
    """The pages' test (top_prob_of_a_sure_row) and closed forms: n equal entries give 1/n;
    entries more than 20 below the top do not count, entries just within do."""
    lg = np.full(100, -30.0, np.float32)
    lg[7] = 30.0
    assert O.top_prob(lg) > 0.999
    assert abs(O.top_prob(np.array([1.0, 1.0], np.float32)) - 0.5) < 1e-5
    assert O.top_prob(np.zeros(8, np.float32)) == np.float32(0.125)
    assert O.top_prob(np.array([0.0, -25.0], np.float32)) == np.float32(1.0)
    # 100000 entries at -20.5 hold 1.25e-4 of a full softmax's mass; top_prob skips them all
    assert O.top_prob(np.concatenate([[0.0], np.full(100_000, -20.5)]).astype(np.float32)) == np.float32(1.0)
    assert O.top_prob(np.array([0.0, -19.0], np.float32)) == np.float32(1.0 / (1.0 + math.exp(-19.0)))
    assert O.top_prob(np.array([3.0, 3.0 - math.log(3.0)], np.float32)) == pytest.approx(0.75, rel=1e-6)


def test_exit_rate_reads_out_while_exits_are_common_and_one_in_eight_after():
    """ExitRate starts at 1.0; each read-out that stays multiplies the rate by 0.9, so the
    first 10 tokens read out (0.9^9 >= 0.35 > 0.9^10), then only tokens 16, 24, ... do; exits
    raise the rate by a tenth of its gap to 1."""
    e = O.ExitRate()
    pattern = []
    for _ in range(24):
        p = e.probe()
        pattern.append(p)
        if p:
            e.note(False)
    assert pattern == [True] * 10 + [False] * 5 + [True] + [False] * 7 + [True]
    assert abs(e.rate - 0.9 ** 12) < 1e-6
    r = e.rate
    e.note(True)
    assert abs(e.rate - (r + 0.1 * (1 - r))) < 1e-7


@pytest.mark.parametrize("kv_mode", ["last_loop", "per_loop"])
def test_a_gated_token_makes_one_pass_when_it_exits_and_two_when_it_stays(kv_mode):
    """th = 0 ends every read-out token after one pass: logits, hidden rows and KV rows are a
    loops=1 token's. th = 2 (above any probability) sends every token to a second pass: they
    are a loops=2 token's, read-out or not (the second read-out replaces the first one's
    output-layer rows)."""
    cfg = micro(kv_mode=kv_mode)
    w = synth.weights(cfg, 24)
    ids = [(i * 7 + 3) % 11 for i in range(30)]
    for th, loops in ((0.0, 1), (2.0, 2)):
        o = O.DoryOracle(cfg, w)
        a, b = O.SeqState(), O.SeqState()
        o.forward_chunk(a, ids[:6], 0, 2, "last")
        o.forward_chunk(b, ids[:6], 0, 2, "last")
        probes = 0
        for i in ids[6:]:
            tokens_before = a.exits.tokens
            la, ha = o.forward_chunk(a, [i], a.pos, 2, "last", gate=th)
            lb, hb = o.forward_chunk(b, [i], b.pos, loops, "last")
            probes += a.exits.tokens - tokens_before
            assert np.max(np.abs(la - lb)) < 1e-12 and np.max(np.abs(ha - hb)) < 1e-12
        assert a.gate_tokens == 24 and a.gate_one == (24 if th == 0.0 else 0)
        assert a.slots.keys() == b.slots.keys()
        for key in a.slots:
            assert a.slots[key].positions == b.slots[key].positions
            for p in a.slots[key].positions:
                assert np.allclose(a.slots[key].k[p], b.slots[key].k[p], atol=1e-12)


# ------------------------------------------------------------------------------------------
# planted mistakes: each pin above must catch a plausible slip in the oracle
# ------------------------------------------------------------------------------------------


def test_a_wrong_rotation_sign_is_caught(monkeypatch):
    def bad(x, cs, sn):
        half = x.shape[-1] // 2
        a, b = x[..., :half], x[..., half:]
        return np.concatenate([a * cs + b * sn, b * cs - a * sn], axis=-1)

    monkeypatch.setattr(O, "rotate_half_split", bad)
    with pytest.raises(AssertionError):
        test_rope_is_a_complex_rotation_of_half_split_pairs()
    with pytest.raises(AssertionError):
        test_oracle_equals_dense_brute_force(4)


def test_a_dropped_residual_normalisation_is_caught(monkeypatch):
    monkeypatch.setattr(O, "residual", lambda x, out, a: O.justnorm(x) + a * (O.justnorm(out) - O.justnorm(x)))
    with pytest.raises(AssertionError):
        test_oracle_equals_dense_brute_force(4)


def test_an_off_by_one_window_is_caught(monkeypatch):
    orig = O.Slot.attend

    def bad(self, qg, kh, p, window):
        return orig(self, qg, kh, p, None if window is None else window + 1)

    monkeypatch.setattr(O.Slot, "attend", bad)
    with pytest.raises(AssertionError):
        test_windowed_attend_equals_masked_full_row()


def test_half_to_even_rounding_is_caught(monkeypatch):
    monkeypatch.setattr(O, "round_half_away", lambda v: np.round(np.asarray(v, np.float32)))
    with pytest.raises(AssertionError):
        test_round_half_away_from_zero()


def test_a_freeze_at_the_64th_row_is_caught(monkeypatch):
    monkeypatch.setattr(O, "KV_COL_WARMUP", 63)
    with pytest.raises(AssertionError):
        test_freeze_comes_at_the_65th_append_and_col_is_the_rms()


def test_a_freeze_sum_in_f64_is_caught(monkeypatch):
    def f64_freeze(codes, scales, group):
        n, hd = codes.shape
        rows = codes.astype(np.float64) * np.repeat(scales, group, axis=1)[:, :hd]
        col = np.maximum(np.sqrt(np.sum(rows * rows, axis=0) / n), 1e-6).astype(np.float32)
        return col, codes, scales

    monkeypatch.setattr(O, "freeze_field", f64_freeze)
    with pytest.raises(AssertionError):
        test_freeze_sums_the_squares_in_f32_in_row_order()


def test_a_rollback_that_keeps_the_dropped_rows_is_caught(monkeypatch):
    def bad(self, st, n):
        st.pos = min(st.pos, n)

    monkeypatch.setattr(O.DoryOracle, "rollback", bad)
    with pytest.raises(AssertionError):
        test_rollback_keeps_the_prefix_a_new_turn_extends()


def test_a_top_prob_that_counts_every_entry_is_caught(monkeypatch):
    def full_softmax(lg):
        lg = np.asarray(lg, np.float64)
        return np.float32(1.0 / np.sum(np.exp(lg - lg.max())))

    monkeypatch.setattr(O, "top_prob", full_softmax)
    with pytest.raises(AssertionError):
        test_top_prob_of_a_sure_row_and_of_ties()


def test_an_exit_rate_that_never_stops_reading_out_is_caught(monkeypatch):
    monkeypatch.setattr(O.ExitRate, "probe", lambda self: True)
    with pytest.raises(AssertionError):
        test_exit_rate_reads_out_while_exits_are_common_and_one_in_eight_after()
